"""Shared test helpers: tolerance checks and bf16 bit conversions."""
import os

import numpy as np
import torch

# Acceptance for fp32 attention output vs the double oracle:
# max |err| <= 2e-3 absolute AND <= 1e-2 * max|V| over the values read.
ATOL = 2e-3
VREL = 1e-2


def bits(t):
    """bf16 tensor (any device) -> uint16 numpy bits on the host."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def vmax_abs(v_bits, lens):
    vf = torch.from_numpy(v_bits.view(np.int16)).view(torch.bfloat16).float()
    m = 0.0
    for b, n in enumerate(lens):
        if n > 0:
            m = max(m, float(vf[b, :, :n].abs().max()))
    return m


def assert_close(out, ref, v_bits, lens, rows=None):
    """out: fp32 torch/numpy [B,Hq,D]; ref: float64 numpy; rows: optional
    (b, h) list restricting the comparison."""
    o = out.detach().cpu().numpy() if isinstance(out, torch.Tensor) else out
    o = o.astype(np.float64)
    if rows is not None:
        idx = np.asarray(rows)
        o = o[idx[:, 0], idx[:, 1]]
        ref = ref[idx[:, 0], idx[:, 1]]
    assert np.all(np.isfinite(o)), "non-finite output"
    err = float(np.abs(o - ref).max()) if o.size else 0.0
    bound = min(ATOL, VREL * vmax_abs(v_bits, lens)) if max(lens) > 0 else ATOL
    assert err <= bound, "max|err| %.3g > bound %.3g" % (err, bound)
    return err


def oracle_threads():
    return max(1, min(64, os.cpu_count() or 1))
