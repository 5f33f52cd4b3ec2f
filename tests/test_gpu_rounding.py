"""The oracle's fp32 -> bf16 rounding (round to nearest, ties to even) pinned
exhaustively against the device: all 2^32 fp32 bit patterns, converted on the
GPU by torch's CUDA float->bfloat16 cast (a library conversion, round to
nearest even) and by the oracle on the CPU.  Every non-NaN pattern must give
the same bits; a NaN must stay a NaN on both sides (each side has its own
NaN payload rule, pinned elsewhere)."""
import numpy as np
import pytest
import torch

import oracle

from gpu_util import DEV

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def test_oracle_bf16_rounding_matches_the_device_on_all_fp32_patterns():
    assert torch.cuda.is_available()
    oracle.build()
    step = 1 << 28
    checked = 0
    for base in range(0, 1 << 32, step):
        p = torch.arange(base, base + step, dtype=torch.int64, device=DEV)
        p = torch.where(p >= (1 << 31), p - (1 << 32), p).to(torch.int32)
        dev = p.view(torch.float32).to(torch.bfloat16).view(torch.int16).cpu().numpy().view(np.uint16)
        del p
        pats = np.arange(base, base + step, dtype=np.uint64).astype(np.uint32)
        ref = oracle.round_bf16_array(pats)
        nan_in = ((pats & 0x7f800000) == 0x7f800000) & ((pats & 0x007fffff) != 0)
        ok = nan_in | (dev == ref)
        if not ok.all():
            i = int(np.nonzero(~ok)[0][0])
            raise AssertionError("pattern 0x%08x: device 0x%04x, oracle 0x%04x" % (int(pats[i]), int(dev[i]),
                                                                                  int(ref[i])))
        dev_nan = ((dev & 0x7f80) == 0x7f80) & ((dev & 0x007f) != 0)
        ref_nan = ((ref & 0x7f80) == 0x7f80) & ((ref & 0x007f) != 0)
        assert (dev_nan[nan_in]).all() and (ref_nan[nan_in]).all()
        checked += int((~nan_in).sum())
    assert checked == (1 << 32) - 2 * ((1 << 23) - 1)  # every pattern except the NaNs
