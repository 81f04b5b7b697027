"""ctypes binding of include/dspark.h — argument marshalling only.

The structs and functions mirror the C ABI one to one and keep its names.  Every
step of the path runs in the CUDA library: if `_lib/libdspark.so` is missing the
first call raises, there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_double, c_float, c_int32, c_size_t, c_uint32, c_uint64, c_void_p

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libdspark.so")

DSPARK_OK = 0
DSPARK_INVALID_ARG = 1
DSPARK_UNSUPPORTED = 2
DSPARK_CUDA_ERROR = 3
DSPARK_TIMEOUT = 4
DSPARK_BAD_INPUT = 5

DSPARK_BF16 = 0
DSPARK_F32 = 1

DSPARK_RESIDUAL_INVERSE_CDF = 0
DSPARK_RESIDUAL_REJECTION = 1
DSPARK_RESIDUAL_TRIALS = 256

DSPARK_HEAD_MARKOV = 0
DSPARK_HEAD_RNN = 1

DSPARK_SCHED_OFF = 0
DSPARK_SCHED_GREEDY = 1
DSPARK_SCHED_ASYNC_TOPK = 2

DSPARK_MAX_GAMMA = 32
DSPARK_MAX_RANK = 1024
DSPARK_MAX_SCHED_KEYS = 65536
DSPARK_MAX_VOCAB = 2097152
DSPARK_STS_MAX_SAMPLES = 8388607
DSPARK_STS_MAX_TABLE = 16384

EXPORTED = ("dspark_workspace_size", "dspark_workspace_init", "dspark_read_error", "dspark_draft_sample",
            "dspark_schedule", "dspark_verify", "dspark_status_string", "dspark_version", "dspark_launch_count",
            "dspark_last_cuda_error", "dspark_schedule_noalloc", "dspark_sts_fit_workspace_size", "dspark_sts_fit",
            "dspark_pack_rows", "dspark_draft_and_schedule")


class dspark_dims(ctypes.Structure):
    _fields_ = [("B", c_int32), ("gamma", c_int32), ("V", c_int32), ("r", c_int32), ("H", c_int32),
                ("dtype", c_int32)]


class dspark_draft_args(ctypes.Structure):
    _fields_ = [("dims", dspark_dims), ("U", c_void_p), ("W1", c_void_p), ("W2", c_void_p), ("h", c_void_p),
                ("w", c_void_p), ("anchor", c_void_p), ("temp", c_void_p), ("req_id", c_void_p),
                ("seed", c_uint64), ("tokens", c_void_p), ("pd_rows", c_void_p), ("pd_tok", c_void_p),
                ("conf_logit", c_void_p), ("conf", c_void_p), ("W_rnn", c_void_p), ("head", c_int32),
                ("pd_stat", c_void_p)]


class dspark_sched_args(ctypes.Structure):
    _fields_ = [("B", c_int32), ("gamma", c_int32), ("mode", c_int32), ("conf_logit", c_void_p),
                ("sts_temp", c_void_p), ("sps", c_void_p), ("anchor", c_void_p), ("tokens", c_void_p),
                ("ell", c_void_p), ("offsets", c_void_p), ("flat_tok", c_void_p), ("mark_req", c_void_p),
                ("mark_pos", c_void_p), ("n_verify", c_void_p), ("n_verify_host", c_void_p),
                ("theta_best", c_void_p), ("surv", c_void_p), ("conf_logit_prev", c_void_p)]


class dspark_verify_args(ctypes.Structure):
    _fields_ = [("dims", dspark_dims), ("target_logits", c_void_p), ("offsets", c_void_p), ("ell", c_void_p),
                ("tokens", c_void_p), ("pd_rows", c_void_p), ("pd_tok", c_void_p), ("temp", c_void_p),
                ("req_id", c_void_p), ("seed", c_uint64), ("n_accept", c_void_p), ("out_tok", c_void_p),
                ("n_out", c_void_p), ("commit_cap", c_void_p), ("residual_mode", c_int32), ("U", c_void_p),
                ("W1", c_void_p), ("W2", c_void_p), ("anchor", c_void_p), ("pd_stat", c_void_p)]


class dspark_pack_args(ctypes.Structure):
    _fields_ = [("V", c_int32), ("dtype", c_int32), ("rows_per_request", c_int32), ("max_rows", c_int32),
                ("n_src_rows", ctypes.c_int64), ("src", c_void_p), ("mark_req", c_void_p), ("mark_pos", c_void_p),
                ("n_rows", c_void_p), ("dst", c_void_p)]


class dspark_sts_fit_args(ctypes.Structure):
    _fields_ = [("N", c_int32), ("gamma", c_int32), ("n_grid", c_int32), ("n_bins", c_int32),
                ("conf_logit", c_void_p), ("accept_len", c_void_p), ("grid", c_void_p), ("sts_temp", c_void_p),
                ("grid_index", c_void_p), ("ece", c_void_p)]


_lib = None


def load() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"dspark CUDA library not built ({LIB_PATH} missing); run "
                           "`python -m draft_sampling_lossless_markov_gb300.build` or __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    lib.dspark_workspace_size.argtypes = [POINTER(dspark_dims), POINTER(c_size_t)]
    lib.dspark_workspace_init.argtypes = [c_void_p, c_size_t, c_void_p]
    lib.dspark_read_error.argtypes = [c_void_p, POINTER(c_int32), POINTER(c_int32), c_void_p]
    lib.dspark_draft_sample.argtypes = [POINTER(dspark_draft_args), c_void_p, c_size_t, c_void_p]
    lib.dspark_schedule.argtypes = [POINTER(dspark_sched_args), c_void_p, c_size_t, c_void_p]
    lib.dspark_draft_and_schedule.argtypes = [POINTER(dspark_draft_args), POINTER(dspark_sched_args), c_void_p,
                                              c_size_t, c_void_p]
    lib.dspark_verify.argtypes = [POINTER(dspark_verify_args), c_void_p, c_size_t, c_void_p]
    lib.dspark_schedule_noalloc.argtypes = [POINTER(dspark_sched_args), c_void_p]
    lib.dspark_sts_fit_workspace_size.argtypes = [c_int32, c_int32, c_int32, c_int32, POINTER(c_size_t)]
    lib.dspark_sts_fit.argtypes = [POINTER(dspark_sts_fit_args), c_void_p, c_size_t, c_void_p]
    lib.dspark_pack_rows.argtypes = [POINTER(dspark_pack_args), c_void_p, c_void_p]
    for f in ("dspark_workspace_size", "dspark_workspace_init", "dspark_read_error", "dspark_draft_sample",
              "dspark_schedule", "dspark_verify", "dspark_schedule_noalloc", "dspark_sts_fit_workspace_size",
              "dspark_sts_fit", "dspark_pack_rows", "dspark_draft_and_schedule"):
        getattr(lib, f).restype = c_int32
    lib.dspark_status_string.argtypes = [c_int32]
    lib.dspark_status_string.restype = c_char_p
    lib.dspark_version.argtypes = []
    lib.dspark_version.restype = c_char_p
    lib.dspark_launch_count.argtypes = []
    lib.dspark_launch_count.restype = c_uint64
    lib.dspark_last_cuda_error.argtypes = []
    lib.dspark_last_cuda_error.restype = c_int32
    _lib = lib
    return lib


def dspark_status_string(s: int) -> str:
    return load().dspark_status_string(s).decode()


def dspark_version() -> str:
    return load().dspark_version().decode()


def dspark_launch_count() -> int:
    return int(load().dspark_launch_count())


def dspark_last_cuda_error() -> int:
    return int(load().dspark_last_cuda_error())


def dspark_workspace_size(dims: dspark_dims) -> tuple[int, int]:
    n = c_size_t(0)
    st = load().dspark_workspace_size(ctypes.byref(dims), ctypes.byref(n))
    return st, n.value


def dspark_workspace_init(workspace: int, nbytes: int, stream: int) -> int:
    return load().dspark_workspace_init(c_void_p(workspace), nbytes, c_void_p(stream))


def dspark_read_error(workspace: int, stream: int) -> tuple[int, int, int]:
    code, detail = c_int32(0), c_int32(0)
    st = load().dspark_read_error(c_void_p(workspace), ctypes.byref(code), ctypes.byref(detail), c_void_p(stream))
    return st, code.value, detail.value


def dspark_draft_sample(args: dspark_draft_args, workspace: int, nbytes: int, stream: int) -> int:
    return load().dspark_draft_sample(ctypes.byref(args), c_void_p(workspace), nbytes, c_void_p(stream))


def dspark_schedule(args: dspark_sched_args, workspace: int, nbytes: int, stream: int) -> int:
    return load().dspark_schedule(ctypes.byref(args), c_void_p(workspace), nbytes, c_void_p(stream))


def dspark_draft_and_schedule(dargs: dspark_draft_args, sargs: dspark_sched_args, workspace: int, nbytes: int,
                              stream: int) -> int:
    """dspark_draft_sample then dspark_schedule in one call that may overlap them."""
    return load().dspark_draft_and_schedule(ctypes.byref(dargs), ctypes.byref(sargs), c_void_p(workspace), nbytes,
                                            c_void_p(stream))


def dspark_schedule_noalloc(args: dspark_sched_args, stream: int) -> int:
    """dspark_schedule without a workspace: scratch in a fixed 1 MiB array inside
    the library, for callers that cannot allocate device memory."""
    return load().dspark_schedule_noalloc(ctypes.byref(args), c_void_p(stream))


def dspark_verify(args: dspark_verify_args, workspace: int, nbytes: int, stream: int) -> int:
    return load().dspark_verify(ctypes.byref(args), c_void_p(workspace), nbytes, c_void_p(stream))


def dspark_sts_fit_workspace_size(N: int, gamma: int, n_grid: int, n_bins: int) -> tuple[int, int]:
    n = c_size_t(0)
    st = load().dspark_sts_fit_workspace_size(N, gamma, n_grid, n_bins, ctypes.byref(n))
    return st, n.value


def dspark_sts_fit(args: dspark_sts_fit_args, workspace: int, nbytes: int, stream: int) -> int:
    return load().dspark_sts_fit(ctypes.byref(args), c_void_p(workspace), nbytes, c_void_p(stream))


def dspark_pack_rows(args: dspark_pack_args, workspace: int, stream: int) -> int:
    return load().dspark_pack_rows(ctypes.byref(args), c_void_p(workspace) if workspace else None, c_void_p(stream))
