"""q4adamw_grad_nonfinite: the optional count of NaN / +-inf BF16 gradients.

The count is a plain definition (exponent bits all ones), checked against
numpy's isfinite on the same BF16 values: special values planted in whole
and ragged tensors (inside 16-byte runs and in tails), the largest finite
BF16 and subnormals not counted, an all-finite list giving 0, and a repeated
call giving the same count (the call zeroes its word first).
"""
import numpy as np
import pytest
import torch

import bit_quantized_adamw_q4adamw_b300 as q4
from bit_quantized_adamw_q4adamw_b300 import workloads as W

pytestmark = pytest.mark.gpu


def test_nonfinite_count_matches_numpy():
    shapes = [(4096,), (3, 129), (5,), (0,), (1000,), (128 * 7 + 3,)]
    w = W.custom("nf", shapes, "zip_sr")
    st = q4.Q4State(w.tensors, "zip_sr")
    rng = np.random.default_rng(3)
    want = 0
    for i, s in enumerate(w.tensors):
        g = rng.normal(0, 1e-3, s.numel).astype(np.float32)
        if s.numel:
            k = rng.choice(s.numel, size=min(s.numel, 7), replace=False)
            g[k[: len(k) // 3]] = np.nan
            g[k[len(k) // 3: 2 * len(k) // 3]] = np.inf
            g[k[2 * len(k) // 3:]] = -np.inf
            g[(k[0] + 1) % s.numel] = 3.3895314e38     # largest finite BF16: not counted
        t = torch.from_numpy(g).to(torch.bfloat16)
        want += int((~np.isfinite(t.float().numpy())).sum())
        st.view(i, "grad").copy_(t)
    out = torch.zeros(1, dtype=torch.int64, device="cuda")
    for _ in range(2):
        q4.q4adamw_grad_nonfinite(st.descs, out, st.workspace)
        torch.cuda.synchronize()
        assert int(out.item()) == want and want > 10
    # all finite (subnormal BF16 included): 0
    for i, s in enumerate(w.tensors):
        st.view(i, "grad").copy_(torch.full((s.numel,), 1e-40, dtype=torch.float32).to(torch.bfloat16))
    q4.q4adamw_grad_nonfinite(st.descs, out, st.workspace)
    torch.cuda.synchronize()
    assert int(out.item()) == 0
