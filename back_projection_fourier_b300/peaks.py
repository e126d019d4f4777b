"""Measured on-chip peaks of this GPU (binding of libtp_peaks.so, include/tp_peaks.h).

``measure()`` runs each microbenchmark of the on-chip units that bound the projection
kernels -- the L1 data pipe (coalesced loads and random 8- / 32-byte gathers), shared-memory
read-modify-writes and atomics, L2 vector reductions and the FP32 pipe -- on the current
device, times each launch with CUDA events on one stream, and returns the best rate of three
launches sized to about two milliseconds each.  The benchmark divides the kernels'
algorithmic work by these rates.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import torch

LIB_PATH = Path(__file__).resolve().parent / "libtp_peaks.so"

KINDS = {"l1_load": 0, "l1_gather8": 1, "l1_gather32": 2, "smem_rmw": 3, "smem_rmw_random": 4,
         "smem_red": 5, "l2_red": 6, "fma": 7}
UNITS = {"l1_load": "loads of 16 B", "l1_gather8": "loads of 8 B", "l1_gather32": "loads of 32 B",
         "smem_rmw": "float2 read-modify-writes", "smem_rmw_random": "float2 read-modify-writes",
         "smem_red": "float atomic adds", "l2_red": "red.global.add.v2.f32", "fma": "flop"}


def _lib() -> ctypes.CDLL:
    if not LIB_PATH.exists():
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m back_projection_fourier_b300.build`")
    L = ctypes.CDLL(str(LIB_PATH))
    L.tp_peak_scratch_bytes.restype = ctypes.c_size_t
    L.tp_peak_run.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int,
                              ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(ctypes.c_double),
                              ctypes.POINTER(ctypes.c_double)]
    L.tp_peak_run.restype = ctypes.c_int
    return L


def measure(device=None, target_ms: float = 2.0, repeats: int = 3) -> dict:
    """{kind: {"ops_per_s", "bytes_per_s", "ms", "unit"}} on `device` (default: current)."""
    L = _lib()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    need = int(L.tp_peak_scratch_bytes())
    scratch = torch.zeros(need + 256, dtype=torch.uint8, device=dev)
    base = scratch.data_ptr()
    ptr = ctypes.c_void_p((base + 255) // 256 * 256)
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    ops, nbytes = ctypes.c_double(), ctypes.c_double()
    ctas = 4 * sms
    out = {"sms": sms, "ctas": ctas}

    def run(kind, iters):
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        rc = L.tp_peak_run(kind, ptr, need, ctas, iters, sp, ctypes.byref(ops), ctypes.byref(nbytes))
        t1.record(stream)
        if rc != 0:
            raise RuntimeError(f"tp_peak_run({kind}) returned {rc}")
        torch.cuda.synchronize(dev)
        return t0.elapsed_time(t1), ops.value, nbytes.value

    for name, kind in KINDS.items():
        iters = 64
        ms, _, _ = run(kind, iters)                  # first launch: loads the module, warms up
        ms, _, _ = run(kind, iters)
        iters = max(16, min(1 << 20, int(iters * target_ms / max(ms, 1e-3))))
        best = None
        for _ in range(repeats):
            ms, o, b = run(kind, iters)
            if best is None or ms < best[0]:
                best = (ms, o, b)
        ms, o, b = best
        out[name] = {"ops_per_s": o / (ms * 1e-3), "bytes_per_s": b / (ms * 1e-3), "ms": ms,
                     "iters": iters, "unit": UNITS[name]}
    return out
