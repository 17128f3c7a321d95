"""Build and load the in-tree CUDA library (``libtopk_ragged.so``).

The library is compiled for GB300 only (``sm_103a``) with nvcc and loaded with
ctypes.  There is no fallback: if the library is missing or cannot be loaded,
every call raises.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT_DIR = os.path.dirname(PKG_DIR)
SRC = os.path.join(PKG_DIR, "csrc", "topk_ragged.cu")
HEADER = os.path.join(ROOT_DIR, "include", "topk_ragged.h")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libtopk_ragged.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"

# Every symbol include/topk_ragged.h declares.
EXPORTS = (
    "topk_ragged_abi_version",
    "topk_ragged_strerror",
    "topk_ragged_init",
    "topk_ragged",
    "topk_ragged_paged",
    "topk_ragged_stats",
    "topk_ragged_indexer_scores",
    "topk_ragged_indexer",
    "topk_ragged_indexer_static",
    "topk_ragged_device_status",
    "topk_ragged_wait_probe",
    "topk_ragged_launch_info",
)

_lock = threading.Lock()
_lib = None


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA library in-tree; returns its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    csrc = os.path.dirname(SRC)
    newest = max([os.path.getmtime(HEADER)] + [os.path.getmtime(os.path.join(csrc, f))
                                                for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h"))])
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= newest:
        return LIB_PATH
    tmp = f"{LIB_PATH}.tmp{os.getpid()}"
    cmd = [nvcc(), ARCH, "-lineinfo", "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-cudart", "shared", "-I" + os.path.join(ROOT_DIR, "include"), SRC, "-o", tmp]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


class TopkError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({strerror(status)})")
        self.status = status


class LaunchInfo(ctypes.Structure):
    _fields_ = [("threads", ctypes.c_int32), ("cluster", ctypes.c_int32),
                ("stage_cap", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("grid", ctypes.c_int32), ("launches", ctypes.c_int32)]


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"CUDA library not built: {LIB_PATH} is missing; run "
                "sparse_attention_deterministic_gb300.build() (nvcc, sm_103a)")
        so = ctypes.CDLL(LIB_PATH)
        so.topk_ragged_abi_version.argtypes = []
        so.topk_ragged_abi_version.restype = ctypes.c_int
        so.topk_ragged_strerror.argtypes = [ctypes.c_int]
        so.topk_ragged_strerror.restype = ctypes.c_char_p
        so.topk_ragged_init.argtypes = [ctypes.c_int]
        so.topk_ragged_init.restype = ctypes.c_int
        so.topk_ragged.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                   ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_void_p]
        so.topk_ragged.restype = ctypes.c_int
        so.topk_ragged_paged.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                         ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p]
        so.topk_ragged_paged.restype = ctypes.c_int
        so.topk_ragged_stats.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
        so.topk_ragged_stats.restype = ctypes.c_int
        vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        so.topk_ragged_indexer_scores.argtypes = [vp, vp, vp, vp, i64, vp, vp, vp, i32, f32, vp, i64, vp]
        so.topk_ragged_indexer_scores.restype = ctypes.c_int
        so.topk_ragged_indexer.argtypes = [vp, vp, vp, vp, i64, vp, vp, vp, i32, f32, vp, i64, i32, i32, vp, vp, vp]
        so.topk_ragged_indexer.restype = ctypes.c_int
        so.topk_ragged_indexer_static.argtypes = [vp, vp, vp, vp, i64, vp, vp, vp, i32, f32, i64, i32, i32, vp, vp,
                                                  vp]
        so.topk_ragged_indexer_static.restype = ctypes.c_int
        so.topk_ragged_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_void_p]
        so.topk_ragged_device_status.restype = ctypes.c_int
        so.topk_ragged_wait_probe.argtypes = [ctypes.c_uint32, ctypes.c_void_p]
        so.topk_ragged_wait_probe.restype = ctypes.c_int
        so.topk_ragged_launch_info.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                               ctypes.POINTER(LaunchInfo)]
        so.topk_ragged_launch_info.restype = ctypes.c_int
        _lib = so
        return so


def strerror(status: int) -> str:
    try:
        return lib().topk_ragged_strerror(int(status)).decode()
    except Exception:  # the library itself is missing
        return "unknown"
