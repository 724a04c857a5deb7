"""Worker for the exhaustive 16-bit rounding pin (runs in spawned processes)."""
import numpy as np
import torch

import oracle


def check_range(args):
    """Compare the oracle's binary32 -> 16-bit rounding with numpy (binary16) or
    torch (bfloat16) over bit patterns [lo, hi).  Returns the number of
    mismatches among non-NaN inputs and of NaN inputs that did not give NaN."""
    lo, hi, dtype = args
    torch.set_num_threads(1)
    bits = np.arange(lo, hi, dtype=np.uint64).astype(np.uint32)
    got = oracle.f32_to_16(bits, dtype)
    f = bits.view(np.float32)
    if dtype == oracle.FP16:
        ref = f.astype(np.float16).view(np.uint16)
        exp_mask, man_mask = 0x7C00, 0x03FF
    else:
        ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        exp_mask, man_mask = 0x7F80, 0x007F
    nan_in = np.isnan(f)
    got_nan = ((got & exp_mask) == exp_mask) & ((got & man_mask) != 0)
    bad = int(np.count_nonzero((got != ref) & ~nan_in))
    bad_nan = int(np.count_nonzero(nan_in & ~got_nan))
    return bad, bad_nan
