"""ctypes view of libsrnn.so (the C ABI declared in include/rnn.h).

Argument marshalling only: every computation runs in the CUDA kernels behind
the C ABI.  There is no CPU fallback; loading fails loudly when the library
has not been built.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
# SRNN_BOUNDS_CHECK=1 loads the bounds-check build (libsrnn_bc.so) instead
LIB_PATH = os.path.join(_PKG, "libsrnn_bc.so" if os.environ.get("SRNN_BOUNDS_CHECK") == "1"
                        else "libsrnn.so")

RNN_LSTM, RNN_GRU, RNN_SLSTM = 0, 1, 2
RNN_F32, RNN_BF16 = 0, 1
RNN_FLAG_TRAIN = 1
RNN_FLAG_H_BF16 = 2
RNN_FLAG_TEST_TIMEOUT = 1 << 30
RNN_HOST_DIRECT = -1  # rnn_fwd_host chunk: the kernel reads / writes the mapped host buffers
STATUS = {0: "RNN_OK", 1: "RNN_ERR_INVALID_ARG", 2: "RNN_ERR_UNSUPPORTED",
          3: "RNN_ERR_MISALIGNED", 4: "RNN_ERR_LAUNCH", 5: "RNN_ERR_TIMEOUT",
          6: "RNN_ERR_NO_CLUSTER", 7: "RNN_ERR_SCRATCH_LIMIT", 8: "RNN_ERR_BOUNDS"}
CELLS = {"lstm": RNN_LSTM, "gru": RNN_GRU, "slstm": RNN_SLSTM}
DTYPES = {"f32": RNN_F32, "bf16": RNN_BF16}

# Every symbol include/rnn.h declares (checked by the CPU tests).
EXPORTS = ("rnn_workspace_size", "rnn_stash_size", "rnn_fwd", "rnn_bwd", "rnn_read_status",
           "rnn_sync_floor", "rnn_fwd_config", "rnn_status_str", "rnn_fwd_noalloc",
           "rnn_input_proj", "rnn_stack_workspace_size", "rnn_stack_fwd", "rnn_plan",
           "rnn_fwd_host_workspace_size", "rnn_fwd_host")


class rnn_desc_t(ctypes.Structure):
    _fields_ = [("cell", ctypes.c_int32), ("dtype", ctypes.c_int32), ("T", ctypes.c_int32),
                ("B", ctypes.c_int32), ("NH", ctypes.c_int32), ("Dh", ctypes.c_int32),
                ("flags", ctypes.c_int32), ("cluster", ctypes.c_int32)]


_P = ctypes.c_void_p
_SZ = ctypes.c_size_t
_I = ctypes.c_int
_DESC = ctypes.POINTER(rnn_desc_t)

_SIGS = {
    "rnn_workspace_size": (_SZ, [_DESC, _I]),
    "rnn_stash_size": (_SZ, [_DESC]),
    "rnn_fwd": (_I, [_DESC] + [_P] * 14 + [_SZ, _P]),
    "rnn_bwd": (_I, [_DESC] + [_P] * 17 + [_SZ, _P]),
    "rnn_read_status": (_I, [_P, _P, ctypes.POINTER(_I)]),
    "rnn_sync_floor": (_I, [_DESC, _I, _P, _SZ, _P]),
    "rnn_fwd_config": (_I, [_DESC, ctypes.POINTER(ctypes.c_int32)]),
    "rnn_status_str": (ctypes.c_char_p, [_I]),
    "rnn_fwd_noalloc": (_I, [_DESC] + [_P] * 15),
    "rnn_input_proj": (_I, [ctypes.c_int32] * 3 + [_P] * 5 + [_SZ, _P]),
    "rnn_stack_workspace_size": (_SZ, [_DESC, ctypes.c_int32, ctypes.c_int32]),
    "rnn_stack_fwd": (_I, [_DESC] + [ctypes.c_int32] * 3 + [_P] * 16 + [_SZ, _P]),
    "rnn_plan": (_I, [_DESC, ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]),
    "rnn_fwd_host_workspace_size": (_SZ, [_DESC, ctypes.c_int32]),
    "rnn_fwd_host": (_I, [_DESC, ctypes.c_int32] + [_P] * 13 + [_SZ, _P]),
}

_lib = None


def load() -> ctypes.CDLL:
    """Load libsrnn.so once; raise if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m sequential_rnn_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib
