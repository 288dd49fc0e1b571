"""Comparison helpers shared by the parity tests.

Routing and dispatch are integer results and must match bit for bit; the
layer output must satisfy |got - ref| <= atol + rtol*|ref| elementwise with
atol = 2e-2 and rtol = 1e-2 (bf16 inputs, fp32 accumulation); gates are fp32
on the GPU against fp64 in the oracle.
"""
import hashlib

import numpy as np

from synth import bf16_to_f32

OUT_ATOL = 2e-2
OUT_RTOL = 1e-2
GATE_RTOL = 2e-6


class ParityError(AssertionError):
    pass


def check_equal(name, got, ref):
    got = np.asarray(got)
    ref = np.asarray(ref)
    if got.shape != ref.shape:
        raise ParityError(f"{name}: shape {got.shape} != {ref.shape}")
    bad = np.flatnonzero(got.reshape(-1) != ref.reshape(-1))
    if bad.size:
        i = bad[0]
        raise ParityError(f"{name}: {bad.size} mismatches, first at flat index {i}: "
                          f"{got.reshape(-1)[i]} != {ref.reshape(-1)[i]}")


def check_dispatch(got: dict, ref: dict):
    for key in ("num_padded", "num_dropped"):
        if int(got[key]) != int(ref[key]):
            raise ParityError(f"{key}: {got[key]} != {ref[key]}")
    for key in ("route_kept", "route_pos", "expert_counts", "sorted_route_ids", "block_expert"):
        check_equal(key, got[key], ref[key])


def check_gates(got, ref, rtol=GATE_RTOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    lim = rtol * np.abs(ref) + 1e-7
    if not np.all(err <= lim):
        i = int(np.argmax(err - lim))
        raise ParityError(f"gates: max excess at {i}: {got.reshape(-1)[i]} vs {ref.reshape(-1)[i]}")


def check_outputs(got_bits, ref, atol=OUT_ATOL, rtol=OUT_RTOL):
    """got_bits: bf16 bit patterns; ref: bf16 bit patterns (uint16) or floats."""
    got = bf16_to_f32(np.asarray(got_bits, dtype=np.uint16)).astype(np.float64)
    ref = np.asarray(ref)
    if ref.dtype == np.uint16:
        ref = bf16_to_f32(ref)
    ref = ref.astype(np.float64)
    if got.shape != ref.shape:
        raise ParityError(f"outputs: shape {got.shape} != {ref.shape}")
    err = np.abs(got - ref)
    lim = atol + rtol * np.abs(ref)
    ok = err <= lim
    if not ok.all():
        i = int(np.argmax(err - lim))
        raise ParityError(f"outputs: {int((~ok).sum())} elements out of tolerance, worst flat "
                          f"index {i}: {got.reshape(-1)[i]} vs {ref.reshape(-1)[i]}")
    return float(err.max()) if err.size else 0.0


def digest(*arrays) -> str:
    m = hashlib.sha256()
    for a in arrays:
        m.update(np.ascontiguousarray(a).tobytes())
    return m.hexdigest()[:16]
