"""Shared helpers for the parity tests: device transfer of bf16 bit patterns and
the layer specification's tolerance (relative Frobenius error <= 5e-3 and
max |delta| <= 2e-2 * max |ref|)."""
import numpy as np

import synth

REL_FROB = 5e-3
MAX_ABS_FRAC = 2e-2


def close(got, ref, rel=REL_FROB, max_frac=MAX_ABS_FRAC):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    nref = np.linalg.norm(ref)
    err = np.linalg.norm(got - ref)
    mx = np.abs(ref).max() if ref.size else 0.0
    dmax = np.abs(got - ref).max() if ref.size else 0.0
    ok = (err <= rel * max(nref, 1e-30)) and (dmax <= max_frac * max(mx, 1e-30))
    return ok, {"rel_frob": err / max(nref, 1e-30), "max_abs": dmax, "max_ref": mx}


def assert_close(got, ref, what=""):
    ok, info = close(got, ref)
    assert ok, f"{what}: {info}"


def to_dev(a, torch, device="cuda"):
    """uint16 bf16 bit patterns -> torch.bfloat16 on the device."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def from_dev_bits(t):
    """torch bf16/int16/uint8/int32 device tensor -> numpy with bf16 as uint16 bits."""
    import torch
    if t.dtype == torch.bfloat16:
        return t.cpu().view(torch.int16).numpy().view(np.uint16)
    return t.cpu().numpy()


def from_dev_f32(t):
    import torch
    if t.dtype == torch.bfloat16:
        return synth.bf16_bits_to_f32(from_dev_bits(t))
    return t.float().cpu().numpy()
