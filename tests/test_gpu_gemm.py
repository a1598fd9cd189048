"""The tcgen05 GEMM (all tilings, all epilogues, fp16 and bf16 operands) against
float64 matmul of the same operand values."""

import pytest
import torch

import chunked_prefill_hybrid_sar_gb300 as sar
import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(autouse=True)
def no_device_flags():
    """Every GEMM test ends with the kernels' device status read back: a
    bounded wait that gave up or a bounds check that fired fails the test."""
    sar.op_sync_status()
    yield
    sar.op_sync_status()


def operands(M, N, K, seed=0, dtype=torch.float16):
    g = synth.generator(seed)
    a = synth.normal(g, (M, K), dtype=torch.bfloat16).to(dtype)
    w = synth.normal(g, (N, K), 0.05, dtype=torch.bfloat16).to(dtype)
    r = synth.normal(g, (M, N), dtype=torch.float32)
    return a, w, r


def close(got, ref, dtype=torch.bfloat16, rel_tol=6e-3):
    """Output rounded once to the storage type: half an ulp relative, plus accumulation noise."""
    got = got.double().cpu()
    ulp = 2 ** -8 if dtype == torch.bfloat16 else 2 ** -11
    err = (got - ref).abs().max().item()
    scale = ref.abs().max().item()
    rel = ((got - ref).norm() / ref.norm()).item()
    assert rel <= rel_tol and err <= ulp * scale + 1e-3, (rel, err, scale)


VARIANTS = {
    "auto": sar.SAR_GEMM_AUTO,
    "m128n128": sar.SAR_GEMM_M128_N128,
    "m128n256": sar.SAR_GEMM_M128_N256,
    "m256n128": sar.SAR_GEMM_M256_N128,
    "swap": sar.SAR_GEMM_SWAP,
    "pair256": sar.SAR_GEMM_PAIR_N256,
    "pair128": sar.SAR_GEMM_PAIR_N128,
    "pair192": sar.SAR_GEMM_PAIR_N192,
}

SHAPES = [(1, 256, 256), (16, 512, 256), (65, 768, 512), (128, 256, 1024), (200, 1024, 256),
          (256, 512, 512), (257, 768, 256), (300, 256, 512), (512, 1024, 512)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("dt", list(DTYPES))
def test_gemm_store(M, N, K, variant, dt):
    if variant == "swap" and M > 256:
        pytest.skip("swap tiling holds at most 256 token rows")
    dtype = DTYPES[dt]
    a, w, _ = operands(M, N, K, dtype=dtype)
    c = torch.empty(M, N, dtype=dtype, device=DEV)
    sar.gemm(a.to(DEV), w.to(DEV), c, variant=VARIANTS[variant])
    torch.cuda.synchronize()
    close(c, a.double() @ w.double().T, dtype)


@pytest.mark.parametrize("M", [3, 130, 384])
@pytest.mark.parametrize("variant", ["auto", "m128n256", "swap", "m256n128", "pair256", "pair128", "pair192"])
@pytest.mark.parametrize("dt", list(DTYPES))
def test_gemm_residual_in_place(M, variant, dt):
    """fp32 residual stream: h = h + a . w^T in place, no rounding to 16 bits."""
    if variant == "swap" and M > 256:
        pytest.skip("swap tiling holds at most 256 token rows")
    N, K = 512, 512
    a, w, r = operands(M, N, K, 1, DTYPES[dt])
    h = r.to(DEV).clone()
    sar.gemm(a.to(DEV), w.to(DEV), h, residual=h, epilogue=sar.SAR_EPI_RESIDUAL, variant=VARIANTS[variant])
    torch.cuda.synchronize()
    ref = a.double() @ w.double().T + r.double()
    assert ((h.double().cpu() - ref).abs().max() / ref.abs().max()).item() < 1e-5


def pack_gate_up(wg, wu):
    """Gate and up rows interleaved in blocks of 64 (the library's packed layout)."""
    F, K = wg.shape
    return torch.stack([wg.view(F // 64, 64, K), wu.view(F // 64, 64, K)], 1).reshape(2 * F, K)


@pytest.mark.parametrize("M", [5, 64, 200, 256, 384])
@pytest.mark.parametrize("variant", ["auto", "m128n128", "m128n256", "swap", "m256n128", "pair256", "pair128"])
@pytest.mark.parametrize("dt", list(DTYPES))
def test_gemm_swiglu(M, variant, dt):
    if variant == "swap" and M > 256:
        pytest.skip("swap tiling holds at most 256 token rows")
    dtype = DTYPES[dt]
    F, K = 512, 256
    g = synth.generator(2)
    a = synth.normal(g, (M, K), dtype=torch.bfloat16).to(dtype)
    wg = synth.normal(g, (F, K), 0.05, dtype=torch.bfloat16).to(dtype)
    wu = synth.normal(g, (F, K), 0.05, dtype=torch.bfloat16).to(dtype)
    out = torch.empty(M, F, dtype=dtype, device=DEV)
    sar.gemm(a.to(DEV), pack_gate_up(wg, wu).to(DEV), out, epilogue=sar.SAR_EPI_SWIGLU,
             variant=VARIANTS[variant])
    torch.cuda.synchronize()
    gg = a.double() @ wg.double().T
    uu = a.double() @ wu.double().T
    close(out, gg / (1 + torch.exp(-gg)) * uu, dtype)


@pytest.mark.parametrize("M", [1, 65, 129])
@pytest.mark.parametrize("dt", list(DTYPES))
def test_gemm_f32_head(M, dt):
    N, K = 1024, 512
    a, w, _ = operands(M, N, K, 3, DTYPES[dt])
    c = torch.empty(M, N, dtype=torch.float32, device=DEV)
    sar.gemm(a.to(DEV), w.to(DEV), c, epilogue=sar.SAR_EPI_F32)
    torch.cuda.synchronize()
    ref = a.double() @ w.double().T
    got = c.double().cpu()
    assert ((got - ref).abs().max() / ref.abs().max()).item() < 1e-5


def test_gemm_pair192_refuses_swiglu():
    a = torch.zeros(256, 256, dtype=torch.float16, device=DEV)
    w = torch.zeros(768, 256, dtype=torch.float16, device=DEV)
    out = torch.zeros(256, 384, dtype=torch.float16, device=DEV)
    with pytest.raises(sar.SarError):
        sar.gemm(a, w, out, epilogue=sar.SAR_EPI_SWIGLU, variant=sar.SAR_GEMM_PAIR_N192)


def test_gemm_unsupported_shapes_are_rejected():
    a = torch.zeros(300, 256, dtype=torch.float16, device=DEV)
    w = torch.zeros(256, 256, dtype=torch.float16, device=DEV)
    c = torch.zeros(300, 256, dtype=torch.float16, device=DEV)
    with pytest.raises(sar.SarError):
        sar.gemm(a, w, c, variant=sar.SAR_GEMM_SWAP)
    with pytest.raises(sar.SarError):
        sar.gemm(a[:, :100], w[:, :100], c)


@pytest.mark.parametrize("rows,hidden", [(1, 256), (260, 256), (512, 4096), (3, 7168)])
@pytest.mark.parametrize("dt", list(DTYPES))
def test_rmsnorm_kernel(rows, hidden, dt):
    g = synth.generator(4)
    x = synth.normal(g, (rows, hidden), 2.0)
    gain = 1 + 0.3 * synth.normal(g, (hidden,))
    y = torch.empty(rows, hidden, dtype=DTYPES[dt], device=DEV)
    sar.rmsnorm(x.to(DEV), gain.to(DEV), y, 1e-5)
    torch.cuda.synchronize()
    xd = x.double()
    ref = xd / torch.sqrt((xd * xd).mean(-1, keepdim=True) + 1e-5) * gain.double()
    close(y, ref, DTYPES[dt])


@pytest.mark.parametrize("M,N,K", [(64, 1024, 4096), (300, 1024, 4096), (512, 2048, 8192)])
def test_gemm_residual_split_k_in_place(M, N, K):
    """Long-K residual GEMMs run split-K (K ranges added atomically into the fp32
    residual); the result must equal one full-K accumulation up to fp32 rounding."""
    a, w, r = operands(M, N, K, 5)
    h = r.to(DEV).clone()
    sar.gemm(a.to(DEV), w.to(DEV), h, residual=h, epilogue=sar.SAR_EPI_RESIDUAL)
    torch.cuda.synchronize()
    ref = a.double() @ w.double().T + r.double()
    assert ((h.double().cpu() - ref).abs().max() / ref.abs().max()).item() < 1e-5


def test_gemm_residual_out_of_place_does_not_split():
    M, N, K = 64, 1024, 4096
    a, w, r = operands(M, N, K, 6)
    c = torch.empty(M, N, dtype=torch.float32, device=DEV)
    sar.gemm(a.to(DEV), w.to(DEV), c, residual=r.to(DEV), epilogue=sar.SAR_EPI_RESIDUAL)
    torch.cuda.synchronize()
    ref = a.double() @ w.double().T + r.double()
    assert ((c.double().cpu() - ref).abs().max() / ref.abs().max()).item() < 1e-5


@pytest.mark.parametrize("M,N,K", [(512, 28672, 4096), (512, 4096, 14336), (1000, 6144, 4096)])
def test_gemm_pair_large(M, N, K):
    """CTA-pair tiles at projection shapes: store and split-K residual in place."""
    a, w, r = operands(M, N, K, 9)
    a, w = a.to(DEV), w.to(DEV)
    c = torch.empty(M, N, dtype=torch.float32, device=DEV)
    sar.gemm(a, w, c, epilogue=sar.SAR_EPI_F32, variant=sar.SAR_GEMM_PAIR_N256)
    h = r.to(DEV).clone()
    sar.gemm(a, w, h, residual=h, epilogue=sar.SAR_EPI_RESIDUAL, variant=sar.SAR_GEMM_PAIR_N256)
    torch.cuda.synchronize()
    # products of 16-bit operands are exact; what remains is fp32 accumulation
    # over K terms in the tensor core's order, which grows like sqrt(K)
    tol = max(1e-5, 3e-7 * K ** 0.5)
    ref = a.double().cpu() @ w.double().cpu().T
    assert ((c.double().cpu() - ref).abs().max() / ref.abs().max()).item() < tol
    ref = ref + r.double()
    assert ((h.double().cpu() - ref).abs().max() / ref.abs().max()).item() < tol


@pytest.mark.parametrize("M", [1, 40, 128])
@pytest.mark.parametrize("epi", ["store", "residual", "swiglu", "f32"])
def test_gemm_swap_two_ctas_per_sm(M, epi):
    """Swap tiling with two CTAs per SM (half the stages each) equals the
    one-CTA launch bit for bit; it is refused above 128 token rows."""
    N, K = 2048, 2048
    a, w, r = operands(M, N, K, 10)
    a, w, r = a.to(DEV), w.to(DEV), r.to(DEV)
    epi_id = {"store": sar.SAR_EPI_STORE, "residual": sar.SAR_EPI_RESIDUAL, "swiglu": sar.SAR_EPI_SWIGLU,
              "f32": sar.SAR_EPI_F32}[epi]
    cols = N // 2 if epi == "swiglu" else N
    odt = torch.float32 if epi in ("residual", "f32") else torch.float16

    def run(flag):
        c = torch.full((M, cols), float("nan"), dtype=odt, device=DEV)
        sar.gemm(a, w, c, residual=r if epi == "residual" else None, epilogue=epi_id,
                 variant=sar.SAR_GEMM_SWAP | flag)
        return c

    base, two = run(0), run(sar.SAR_GEMM_TWO_CTAS)
    torch.cuda.synchronize()
    assert torch.equal(base, two)
    with pytest.raises(sar.SarError):
        sar.gemm(torch.zeros(200, K, dtype=torch.float16, device=DEV), w,
                 torch.zeros(200, N, dtype=torch.float16, device=DEV),
                 variant=sar.SAR_GEMM_SWAP | sar.SAR_GEMM_TWO_CTAS)


@pytest.mark.parametrize("M,N,K,variant,flags", [
    (512, 4096, 4096, "pair256", 0),         # the O projection at 512 rows
    (512, 4096, 14336, "pair256", 0),        # the down projection at 512 rows
    (1000, 6144, 4096, "pair128", 0),        # ragged token tiles, an all-padding partner tile
    (300, 1024, 4096, "m128n256", 0),        # single CTAs, ragged rows
    (512, 2048, 8192, "m128n256", 0),        # four token groups, K = 8192
    (100, 192, 320, "m128n128", 0),          # fewer K slabs than CTAs: most shares are empty
])
def test_gemm_stream_k_residual_in_place(M, N, K, variant, flags):
    """Stream-K: every resident CTA (pair) takes an equal run of all tiles' K
    slabs and adds partial tiles atomically; the result equals one full-K
    accumulation up to fp32 rounding."""
    a, w, r = operands(M, N, K, 11)
    h = r.to(DEV).clone()
    sar.gemm(a.to(DEV), w.to(DEV), h, residual=h, epilogue=sar.SAR_EPI_RESIDUAL,
             variant=VARIANTS[variant] | flags | sar.SAR_GEMM_STREAM_K)
    torch.cuda.synchronize()
    ref = a.double() @ w.double().T + r.double()
    tol = max(1e-5, 3e-7 * K ** 0.5)
    assert ((h.double().cpu() - ref).abs().max() / ref.abs().max()).item() < tol


def test_gemm_stream_k_is_refused_where_partial_sums_cannot_add():
    a = torch.zeros(512, 1024, dtype=torch.float16, device=DEV)
    w = torch.zeros(1024, 1024, dtype=torch.float16, device=DEV)
    c16 = torch.zeros(512, 1024, dtype=torch.float16, device=DEV)
    c32 = torch.zeros(512, 1024, dtype=torch.float32, device=DEV)
    r32 = torch.zeros(512, 1024, dtype=torch.float32, device=DEV)
    with pytest.raises(sar.SarError):  # a stored (rounded) output
        sar.gemm(a, w, c16, variant=sar.SAR_GEMM_PAIR_N256 | sar.SAR_GEMM_STREAM_K)
    with pytest.raises(sar.SarError):  # residual out of place
        sar.gemm(a, w, c32, residual=r32, epilogue=sar.SAR_EPI_RESIDUAL,
                 variant=sar.SAR_GEMM_PAIR_N256 | sar.SAR_GEMM_STREAM_K)
    with pytest.raises(sar.SarError):  # swap tiling
        sar.gemm(a[:64], w, c32[:64], residual=c32[:64], epilogue=sar.SAR_EPI_RESIDUAL,
                 variant=sar.SAR_GEMM_SWAP | sar.SAR_GEMM_STREAM_K)
