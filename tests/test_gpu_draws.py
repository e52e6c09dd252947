"""The step's stochastic-rounding draws on the GPU against the oracle's Philox.

q4adamw_draws evaluates the device Philox4x32-10 function the step kernel
uses; every 32-bit word must equal the oracle's (itself pinned to cuRAND's
host Philox4_32_10 generator) for the same (seed, step, tensor id, element,
purpose) -- including element indices across the 2^34 boundary of the
counter's second word, the largest seed, step and tensor id, and starts that
are not a multiple of 4.
"""
import numpy as np
import pytest
import torch

import bit_quantized_adamw_q4adamw_b300 as q4
from oracle import oracle as O

pytestmark = pytest.mark.gpu

CASES = [
    (0, 1, 0, 0, 0, 4096),
    (0, 1, 0, 0, 1, 4096),
    (12345, 7, 3, 1000, 1, 777),
    (2 ** 64 - 1, 2 ** 32 - 1, 2 ** 32 - 1, 5, 0, 300),
    (0xDEADBEEFCAFEF00D, 9001, 290, 2 ** 34 - 6, 1, 20),
    (42, 123456, 17, 8_030_261_248 - 129, 0, 129),
    (7, 2, 1, 3, 1, 1),
]


@pytest.mark.parametrize("seed,step,tid,idx0,purpose,n", CASES)
def test_draws_match_oracle(seed, step, tid, idx0, purpose, n):
    out = torch.empty(n, dtype=torch.int32, device="cuda")
    q4.q4adamw_draws(seed, step, tid, idx0, purpose, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint32)
    want = O.draws(seed, step, tid, idx0, n, purpose)
    assert np.array_equal(got, want), (int(np.argmax(got != want)), got[:4], want[:4])


def test_draws_differ_by_purpose_and_tensor():
    a = torch.empty(1024, dtype=torch.int32, device="cuda")
    b = torch.empty_like(a)
    c = torch.empty_like(a)
    q4.q4adamw_draws(1, 1, 0, 0, 0, a)
    q4.q4adamw_draws(1, 1, 0, 0, 1, b)
    q4.q4adamw_draws(1, 1, 1, 0, 0, c)
    torch.cuda.synchronize()
    assert (a != b).float().mean() > 0.99 and (a != c).float().mean() > 0.99
