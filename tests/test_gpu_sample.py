"""Greedy sampling on the device (sar_sample_greedy): each logits row's
argmax, the lowest index among equal maxima (the serving loop's sampler; the
pages' traces decode greedily to a fixed output length)."""

import dataclasses

import pytest
import torch

import synth
from chunked_prefill_hybrid_sar_gb300 import harness

pytestmark = pytest.mark.gpu


def model_with_vocab(vocab):
    case = synth.tiny_case(0, dtype=torch.bfloat16)
    dims = dataclasses.replace(case["dims"], vocab=vocab)
    _, head, _ = synth.model_weights(0, dims, torch.bfloat16)
    return harness.load_model(dims, case["layers"], head, max_tokens=64, max_decodes=8)


# rows starting on a 16-byte boundary take the float4 scan; logits one float
# past it (offset 1) take the scalar scan
@pytest.mark.parametrize("rows,vocab,offset", [(1, 32000, 0), (65, 32000, 0), (7, 1024, 0), (65, 64000, 0),
                                               (4, 32000, 1), (3, 64, 1)])
def test_argmax_with_planted_ties(rows, vocab, offset):
    m = model_with_vocab(vocab)
    g = torch.Generator().manual_seed(rows * 7 + vocab)
    x = torch.randn(rows, vocab, generator=g)
    for r in range(rows):  # plant the row maximum at several indices
        idx = torch.randperm(vocab, generator=g)[:3]
        x[r, idx] = x[r].max() + 1.0
    buf = torch.zeros(rows * vocab + offset, device="cuda")
    buf[offset:] = x.reshape(-1).cuda()
    out = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
    m.sample_greedy(buf[offset:], rows, out)
    torch.cuda.synchronize()
    m.close()
    assert torch.equal(out.cpu(), x.argmax(dim=1).to(torch.int32))
