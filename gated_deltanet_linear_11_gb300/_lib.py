"""ctypes binding of libgdn.so.  Argument marshalling only: every step runs in the CUDA
kernels behind the C ABI declared in include/gdn.h.  There is no CPU fallback: if the
library is missing or fails to load, every call raises."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libgdn.so")

GDN_BF16, GDN_F32, GDN_I32 = 0, 1, 2
GDN_QK_L2NORM = 0x1
GDN_PREFILL_SIMT = 0x100
GDN_PREFILL_TILES2 = 0x200
GDN_PREFILL_TILES3 = 0x400
GDN_LAYER_FUSED_VCONV = 0x800
GDN_CHECK_INPUTS = 0x1000

STATUS = {
    0: "GDN_OK", 1: "GDN_ERR_NULL", 2: "GDN_ERR_SHAPE", 3: "GDN_ERR_LAYOUT",
    4: "GDN_ERR_DTYPE", 5: "GDN_ERR_SEQLENS", 6: "GDN_ERR_UNSUPPORTED", 7: "GDN_ERR_CUDA",
    8: "GDN_ERR_TIMEOUT", 9: "GDN_ERR_WORKSPACE", 10: "GDN_ERR_INDEX",
    11: "GDN_ERR_NONFINITE",
}

EXPORTS = ("gdn_status_string", "gdn_version", "gdn_conv1d_fwd", "gdn_conv1d_update",
           "gdn_chunk_prefill_workspace_size", "gdn_chunk_prefill",
           "gdn_chunk_prefill_noalloc", "gdn_chunk_prefill_cp_workspace_size",
           "gdn_chunk_prefill_cp", "gdn_chunk_prefill_cp_range_hint",
           "gdn_chunk_prefill_cp_range_hint_for", "gdn_recurrent_decode", "gdn_fused_decode",
           "gdn_layer_prefill", "gdn_selftest_bounded_wait")

NOALLOC_SCRATCH_BYTES = 128 << 20


class GdnTensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("ndim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("shape", ctypes.c_int64 * 4),
                ("stride", ctypes.c_int64 * 4)]


class GdnError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__("%s returned %s" % (where, STATUS.get(code, code)))


_lib = None


def load(path: str = LIB_PATH):
    """Load libgdn.so and declare the signatures.  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libgdn.so not built (%s); run gated_deltanet_linear_11_gb300"
                           ".build.build() -- there is no fallback path" % path)
    lib = ctypes.CDLL(path)
    vp, i32, i64, u32, f32 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                              ctypes.c_uint32, ctypes.c_float)
    tp = ctypes.POINTER(GdnTensor)
    sig = {
        "gdn_status_string": ([i32], ctypes.c_char_p),
        "gdn_version": ([], i32),
        "gdn_conv1d_fwd": ([vp, i64, i32, vp, vp, vp, vp, i32, vp, vp, vp, vp], i32),
        "gdn_conv1d_update": ([vp, i32, i32, vp, vp, vp, i32, vp, vp, vp, vp], i32),
        "gdn_chunk_prefill_workspace_size": ([i32, i64, i32, i32, i32, i32, i32, u32],
                                             ctypes.c_size_t),
        "gdn_chunk_prefill": ([tp, tp, tp, vp, vp, vp, vp, i32, i32, f32, u32, vp, tp, vp,
                               vp, ctypes.c_size_t, vp, vp], i32),
        "gdn_chunk_prefill_noalloc": ([tp, tp, tp, vp, vp, vp, vp, i32, i32, f32, u32, vp,
                                       tp, vp, vp, vp], i32),
        "gdn_chunk_prefill_cp_workspace_size": ([vp, i32, i64, i32, i32, i32, i32, i32, i32],
                                                ctypes.c_size_t),
        "gdn_chunk_prefill_cp": ([tp, tp, tp, vp, vp, vp, vp, i32, i32, f32, u32, i32, vp, tp,
                                  vp, vp, ctypes.c_size_t, vp, vp], i32),
        "gdn_chunk_prefill_cp_range_hint": ([i64, i32], i32),
        "gdn_chunk_prefill_cp_range_hint_for": ([i64, i32, i32], i32),
        "gdn_recurrent_decode": ([tp, tp, tp, vp, vp, vp, i32, vp, f32, u32, tp, vp, vp],
                                 i32),
        "gdn_fused_decode": ([vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, i32, vp,
                              f32, u32, vp, vp, vp], i32),
        "gdn_layer_prefill": ([vp, i64, i32, i32, i32, i32, vp, vp, vp, vp, i32, vp, vp, vp,
                               vp, vp, f32, u32, vp, vp, vp, vp, ctypes.c_size_t, vp, vp,
                               vp], i32),
        "gdn_selftest_bounded_wait": ([vp, vp], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def check(code, where):
    if code != 0:
        raise GdnError(code, where)
