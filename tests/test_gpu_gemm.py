"""The tcgen05 GEMM (all tilings, all epilogues) against float64 matmul of the same bf16 operands."""

import pytest
import torch

import chunked_prefill_hybrid_sar_gb300 as sar
import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


def operands(M, N, K, seed=0):
    g = synth.generator(seed)
    a = synth.normal(g, (M, K), dtype=torch.bfloat16)
    w = synth.normal(g, (N, K), 0.05, dtype=torch.bfloat16)
    r = synth.normal(g, (M, N), dtype=torch.bfloat16)
    return a, w, r


def close(got, ref, rel_tol=6e-3):
    got = got.double().cpu()
    err = (got - ref).abs().max().item()
    scale = ref.abs().max().item()
    rel = ((got - ref).norm() / ref.norm()).item()
    assert rel <= rel_tol and err <= 2 ** -7 * scale + 1e-3, (rel, err, scale)


VARIANTS = {
    "auto": sar.SAR_GEMM_AUTO,
    "m128n128": sar.SAR_GEMM_M128_N128,
    "m128n256": sar.SAR_GEMM_M128_N256,
    "m256n128": sar.SAR_GEMM_M256_N128,
    "swap": sar.SAR_GEMM_SWAP,
}

SHAPES = [(1, 256, 256), (16, 512, 256), (65, 768, 512), (128, 256, 1024), (200, 1024, 256),
          (256, 512, 512), (257, 768, 256), (300, 256, 512), (512, 1024, 512)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("variant", list(VARIANTS))
def test_gemm_bf16(M, N, K, variant):
    if variant == "swap" and M > 256:
        pytest.skip("swap tiling holds at most 256 token rows")
    a, w, _ = operands(M, N, K)
    c = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    sar.gemm(a.to(DEV), w.to(DEV), c, variant=VARIANTS[variant])
    torch.cuda.synchronize()
    close(c, a.double() @ w.double().T)


@pytest.mark.parametrize("M", [3, 130, 384])
@pytest.mark.parametrize("variant", ["auto", "m128n256", "swap"])
def test_gemm_residual_in_place(M, variant):
    if variant == "swap" and M > 256:
        pytest.skip("swap tiling holds at most 256 token rows")
    N, K = 512, 512
    a, w, r = operands(M, N, K, 1)
    h = r.to(DEV).clone()
    sar.gemm(a.to(DEV), w.to(DEV), h, residual=h, epilogue=sar.SAR_EPI_RESIDUAL, variant=VARIANTS[variant])
    torch.cuda.synchronize()
    close(h, a.double() @ w.double().T + r.double())


def pack_gate_up(wg, wu):
    """Gate and up rows interleaved in blocks of 64 (the library's packed layout)."""
    F, K = wg.shape
    return torch.stack([wg.view(F // 64, 64, K), wu.view(F // 64, 64, K)], 1).reshape(2 * F, K)


@pytest.mark.parametrize("M", [5, 64, 200, 256, 384])
@pytest.mark.parametrize("variant", ["auto", "m128n128", "m128n256", "swap", "m256n128"])
def test_gemm_swiglu(M, variant):
    if variant == "swap" and M > 256:
        pytest.skip("swap tiling holds at most 256 token rows")
    F, K = 512, 256
    g = synth.generator(2)
    a = synth.normal(g, (M, K), dtype=torch.bfloat16)
    wg = synth.normal(g, (F, K), 0.05, dtype=torch.bfloat16)
    wu = synth.normal(g, (F, K), 0.05, dtype=torch.bfloat16)
    out = torch.empty(M, F, dtype=torch.bfloat16, device=DEV)
    sar.gemm(a.to(DEV), pack_gate_up(wg, wu).to(DEV), out, epilogue=sar.SAR_EPI_SWIGLU,
             variant=VARIANTS[variant])
    torch.cuda.synchronize()
    gg = a.double() @ wg.double().T
    uu = a.double() @ wu.double().T
    close(out, gg / (1 + torch.exp(-gg)) * uu)


@pytest.mark.parametrize("M", [1, 65, 129])
def test_gemm_f32_head(M):
    N, K = 1024, 512
    a, w, _ = operands(M, N, K, 3)
    c = torch.empty(M, N, dtype=torch.float32, device=DEV)
    sar.gemm(a.to(DEV), w.to(DEV), c, epilogue=sar.SAR_EPI_F32)
    torch.cuda.synchronize()
    ref = a.double() @ w.double().T
    got = c.double().cpu()
    assert ((got - ref).abs().max() / ref.abs().max()).item() < 1e-5


def test_gemm_unsupported_shapes_are_rejected():
    a = torch.zeros(300, 256, dtype=torch.bfloat16, device=DEV)
    w = torch.zeros(256, 256, dtype=torch.bfloat16, device=DEV)
    c = torch.zeros(300, 256, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(sar.SarError):
        sar.gemm(a, w, c, variant=sar.SAR_GEMM_SWAP)
    with pytest.raises(sar.SarError):
        sar.gemm(a[:, :100], w[:, :100], c)


@pytest.mark.parametrize("rows,hidden", [(1, 256), (260, 256), (512, 4096), (3, 7168)])
def test_rmsnorm_kernel(rows, hidden):
    g = synth.generator(4)
    x = synth.normal(g, (rows, hidden), 2.0, dtype=torch.bfloat16)
    gain = (1 + 0.3 * synth.normal(g, (hidden,))).to(torch.bfloat16)
    y = torch.empty_like(x, device=DEV)
    sar.rmsnorm(x.to(DEV), gain.to(DEV), y, 1e-5)
    torch.cuda.synchronize()
    xd = x.double()
    ref = xd / torch.sqrt((xd * xd).mean(-1, keepdim=True) + 1e-5) * gain.double()
    close(y, ref)
