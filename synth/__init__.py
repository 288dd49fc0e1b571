"""Seeded synthetic inputs for the batch-invariant MoE layer.

Only input generation lives here (no routing, dispatch or expert arithmetic),
so both the CUDA path and the CPU checker may draw from it.  The generator is
counter-based (see synth.c): element i of tensor (seed, tensor_id) is a pure
function of (seed, tensor_id, i), identical on host and device.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_SO = os.path.join(_HERE, "libsynth.so")
_GPU_SO = os.path.join(_HERE, "libsynth_gpu.so")

_host = None
_gpu = None


def build(gpu: bool = True) -> None:
    """Compile the host generator (gcc) and, if asked, the device one (nvcc)."""
    src = os.path.join(_HERE, "synth.c")
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-o", _HOST_SO, src])
    if gpu:
        cu = os.path.join(_HERE, "synth_gpu.cu")
        subprocess.check_call([
            "nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared",
            "-Xcompiler", "-fPIC", "-o", _GPU_SO, cu,
        ])


def _host_lib():
    global _host
    if _host is None:
        if not os.path.exists(_HOST_SO):
            build(gpu=False)
        lib = ctypes.CDLL(_HOST_SO)
        lib.synth_normal_bf16.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                                          ctypes.c_uint64, ctypes.c_uint64, ctypes.c_float, ctypes.c_int]
        lib.synth_normal_bf16.restype = None
        lib.synth_uniform_u64.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                                          ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_uniform_u64.restype = None
        _host = lib
    return _host


def _gpu_lib():
    global _gpu
    if _gpu is None:
        if not os.path.exists(_GPU_SO):
            raise RuntimeError("libsynth_gpu.so is not built; run __graft_entry__.build()")
        lib = ctypes.CDLL(_GPU_SO)
        lib.synth_normal_bf16_gpu.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                                              ctypes.c_uint64, ctypes.c_uint64, ctypes.c_float,
                                              ctypes.c_void_p]
        lib.synth_normal_bf16_gpu.restype = ctypes.c_int
        _gpu = lib
    return _gpu


def scale_for_std(std: float) -> float:
    """fp32 multiplier that maps the Irwin-Hall integer to N(0, std^2)."""
    return float(np.float32(std / 65536.0))


def normal_bf16(shape, seed: int, tensor_id: int, std: float, offset: int = 0,
                nthreads: int | None = None) -> np.ndarray:
    """bf16 bit patterns (uint16) of approximately N(0, std^2) values."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.uint16)
    if nthreads is None:
        nthreads = min(32, os.cpu_count() or 1)
    _host_lib().synth_normal_bf16(out.ctypes.data, n, offset, seed, tensor_id,
                                  scale_for_std(std), nthreads)
    return out.reshape(shape)


def uniform_u64(n: int, seed: int, tensor_id: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _host_lib().synth_uniform_u64(out.ctypes.data, n, offset, seed, tensor_id)
    return out


def normal_bf16_device(tensor, seed: int, tensor_id: int, std: float, offset: int = 0,
                       stream: int = 0) -> None:
    """Fill a contiguous torch uint16/bfloat16 CUDA tensor in place on the device."""
    n = tensor.numel()
    rc = _gpu_lib().synth_normal_bf16_gpu(tensor.data_ptr(), n, offset, seed, tensor_id,
                                          scale_for_std(std), stream)
    if rc != 0:
        raise RuntimeError(f"synth_normal_bf16_gpu failed with CUDA error {rc}")


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 exactly."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 bit patterns, nearest-even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)
