"""The attention tolerance of tests/util.py tells a correct kernel from one that loses work.

At the Llama-3-8B drop-4x shape (8,192 kept rows per KV head, 32/8 heads, d 128) the outputs have
a standard deviation near 0.011, so the per-element bound max(1e-2, 2e-2 |oracle|) alone accepts
almost anything. Two plausible kernel mistakes are planted in copies of the oracle's output:
  - four 16-row chunks (64 of the 8,192 kept rows) left out of every head's softmax;
  - the softmax scale 1/sqrt(d) multiplied by 0.95;
both must fail the relative-L2 / tight per-element checks, while the oracle's output rounded to
bf16 (what a correct kernel with fp32 accumulation stores) must pass all three checks. CPU only.
"""
import numpy as np
import pytest
import torch

import oracle as O
from tests.util import attn_errors, assert_attn_close, REL_L2

KEEP, HQ, HKV, D = 8192, 32, 8, 128


@pytest.fixture(scope="module")
def case():
    g = torch.Generator().manual_seed(20261203)
    bf = lambda *s: torch.randn(s, generator=g).to(torch.bfloat16).to(torch.float32).numpy()
    q, k, v = bf(HQ, D), bf(HKV, KEEP, D), bf(HKV, KEEP, D)
    empty = np.zeros((HKV, 0, D), np.float32)
    ref = O.draft_attn(q, k, v, empty, empty)
    return q, k, v, empty, ref


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def test_correct_bf16_output_passes(case):
    q, k, v, empty, ref = case
    assert np.std(ref) < 0.02  # the regime where the per-element floor of 1e-2 is blind
    assert_attn_close(_bf16(ref), ref, "bf16-rounded oracle")


def test_dropped_chunks_fail(case):
    q, k, v, empty, ref = case
    keep = np.ones(KEEP, bool)
    for c in (3, 100, 257, 500):  # four 16-row chunks
        keep[16 * c:16 * c + 16] = False
    bad = _bf16(O.draft_attn(q, k[:, keep], v[:, keep], empty, empty))
    n1, rel, n3, _ = attn_errors(bad, ref)
    assert rel > REL_L2 and n3 > 0, (n1, rel, n3)
    with pytest.raises(AssertionError):
        assert_attn_close(bad, ref, "64 rows dropped")


def test_scaled_softmax_fails(case):
    q, k, v, empty, ref = case
    bad = _bf16(O.draft_attn(0.95 * q, k, v, empty, empty))
    n1, rel, n3, _ = attn_errors(bad, ref)
    assert rel > REL_L2 and n3 > 0, (n1, rel, n3)
    with pytest.raises(AssertionError):
        assert_attn_close(bad, ref, "scale x 0.95")
