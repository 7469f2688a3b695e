"""Comparison helpers for the GPU parity tests (test code only)."""
import numpy as np
import torch

# Final-output tolerance of the layer: relative Frobenius error and max
# absolute error against the oracle.
FINAL_REL_FRO = 1e-2
FINAL_MAX_ABS = 5e-2


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_val(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def e4m3_val(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def rel_fro(got: np.ndarray, ref: np.ndarray) -> float:
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (n if n > 0 else 1.0))


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (np.maximum(e, -126) - 7), 2.0 ** -133)


def assert_bf16_close(got_bits, ref_bits, what, ulps=1, rel=2e-3, floor_rel=1e-5):
    """Element-wise within `ulps` bf16 steps of the reference (plus a floor
    relative to the array's largest magnitude, for cancellation to ~0), and
    relative Frobenius error <= rel."""
    g, r = bf16_val(got_bits), bf16_val(ref_bits)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    tol = ulps * bf16_ulp(r) + floor_rel * np.abs(r).max()
    bad = np.abs(g - r) > tol
    fro = rel_fro(g, r)
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} elements beyond {ulps} ulp; "
                           f"worst {np.abs(g - r).max():.3e}; rel_fro {fro:.2e}")
    assert fro <= rel, f"{what}: rel_fro {fro:.3e} > {rel}"
    return fro, float((g != r).mean())


def assert_final_close(got_bits, ref_bits, what):
    g, r = bf16_val(got_bits), bf16_val(ref_bits)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    fro = rel_fro(g, r)
    mx = float(np.abs(g - r).max()) if g.size else 0.0
    assert fro <= FINAL_REL_FRO and mx <= FINAL_MAX_ABS, f"{what}: rel_fro {fro:.3e}, max_abs {mx:.3e}"
    return fro, mx
