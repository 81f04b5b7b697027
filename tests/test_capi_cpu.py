"""The C-ABI library builds, loads and exports every declared symbol; argument
checks that return before any CUDA call (CPU only: no compute call is made)."""
import ctypes
import os
import re

import pytest

from draft_sampling_lossless_markov_gb300 import build, capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return capi.load()


def _declared():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            names |= set(re.findall(r"DSPARK_API\s+[\w\s\*]+?\b(dspark_\w+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(lib):
    declared = _declared()
    assert {"dspark_draft_sample", "dspark_schedule", "dspark_verify"} <= declared
    for name in declared:
        assert hasattr(lib, name), name
    assert set(capi.EXPORTED) <= declared


def test_status_strings_and_version(lib):
    assert capi.dspark_status_string(capi.DSPARK_OK) == "DSPARK_OK"
    assert capi.dspark_status_string(capi.DSPARK_TIMEOUT) == "DSPARK_TIMEOUT"
    assert capi.dspark_status_string(99) == "DSPARK_UNKNOWN_STATUS"
    assert "sm_103a" in capi.dspark_version()


def test_workspace_size(lib):
    st, n = capi.dspark_workspace_size(capi.dspark_dims(256, 7, 151936, 256, 4096, capi.DSPARK_BF16))
    assert st == capi.DSPARK_OK and n > 0 and n % 256 == 0
    st2, n2 = capi.dspark_workspace_size(capi.dspark_dims(256, 7, 151936, 0, 0, capi.DSPARK_BF16))
    assert st2 == capi.DSPARK_OK and n2 < n
    for bad in (capi.dspark_dims(4, 0, 10, 1, 1, 0), capi.dspark_dims(4, 33, 10, 1, 1, 0),
                capi.dspark_dims(-1, 4, 10, 1, 1, 0), capi.dspark_dims(4, 4, 0, 1, 1, 0),
                capi.dspark_dims(4, 4, 10, 1025, 1, 0), capi.dspark_dims(4, 4, 10, 1, 1, 7)):
        assert capi.dspark_workspace_size(bad)[0] == capi.DSPARK_INVALID_ARG
    assert lib.dspark_workspace_size(None, None) == capi.DSPARK_INVALID_ARG


def test_argument_errors_return_before_any_launch(lib):
    d = capi.dspark_draft_args()
    d.dims = capi.dspark_dims(4, 4, 64, 8, 16, capi.DSPARK_F32)
    # null inputs
    assert capi.dspark_draft_sample(d, 0, 0, 0) == capi.DSPARK_INVALID_ARG
    assert lib.dspark_draft_sample(None, None, 0, None) == capi.DSPARK_INVALID_ARG
    # empty batch: nothing to do, no CUDA call
    d.dims = capi.dspark_dims(0, 4, 64, 8, 16, capi.DSPARK_F32)
    assert capi.dspark_draft_sample(d, 0, 0, 0) == capi.DSPARK_OK
    # misaligned input pointer (checked before the workspace)
    d.dims = capi.dspark_dims(4, 4, 64, 8, 16, capi.DSPARK_F32)
    for f in ("U", "W1", "W2", "h", "w", "anchor", "temp", "req_id", "tokens", "pd_rows", "pd_tok", "conf_logit",
              "conf"):
        setattr(d, f, 0x10000)
    d.U = 0x10004
    assert capi.dspark_draft_sample(d, 0x20000, 1 << 30, 0) == capi.DSPARK_INVALID_ARG
    # workspace too small / misaligned
    d.U = 0x10000
    assert capi.dspark_draft_sample(d, 0x20000, 16, 0) == capi.DSPARK_INVALID_ARG
    assert capi.dspark_draft_sample(d, 0x20010, 1 << 30, 0) == capi.DSPARK_INVALID_ARG

    s = capi.dspark_sched_args()
    s.B, s.gamma, s.mode = 4096, 17, capi.DSPARK_SCHED_GREEDY
    assert capi.dspark_schedule(s, 0, 0, 0) == capi.DSPARK_UNSUPPORTED  # B * gamma > 65536
    s.B, s.gamma = 4, 33
    assert capi.dspark_schedule(s, 0, 0, 0) == capi.DSPARK_INVALID_ARG
    s.gamma, s.mode = 4, 5
    assert capi.dspark_schedule(s, 0, 0, 0) == capi.DSPARK_INVALID_ARG
    s.mode = capi.DSPARK_SCHED_GREEDY
    assert capi.dspark_schedule(s, 0, 0, 0) == capi.DSPARK_INVALID_ARG  # null pointers
    s.B = 0
    assert capi.dspark_schedule(s, 0, 0, 0) == capi.DSPARK_OK
    # asynchronous mode: needs the earlier confidences and the cost table, and
    # one CTA's shared memory
    for f in ("conf_logit", "sts_temp", "sps", "anchor", "tokens", "ell", "offsets", "flat_tok", "mark_req",
              "mark_pos", "n_verify", "theta_best"):
        setattr(s, f, 0x10000)
    s.B, s.gamma, s.mode = 64, 7, capi.DSPARK_SCHED_ASYNC_TOPK
    assert capi.dspark_schedule(s, 0, 0, 0) == capi.DSPARK_INVALID_ARG  # no conf_logit_prev
    s.conf_logit_prev = 0x10000
    s.B = 4096
    assert capi.dspark_schedule(s, 0, 0, 0) == capi.DSPARK_UNSUPPORTED  # 32768 slots
    assert capi.dspark_schedule_noalloc(s, 0) == capi.DSPARK_UNSUPPORTED

    # the combined draft + schedule call: its own consistency checks, then both calls' checks
    d.dims = capi.dspark_dims(64, 7, 64, 8, 16, capi.DSPARK_F32)
    s.B, s.gamma, s.mode, s.conf_logit_prev = 64, 7, capi.DSPARK_SCHED_GREEDY, None
    s.conf_logit, s.tokens, s.anchor = d.conf_logit, d.tokens, d.anchor
    assert lib.dspark_draft_and_schedule(None, ctypes.byref(s), None, 0, None) == capi.DSPARK_INVALID_ARG
    assert lib.dspark_draft_and_schedule(ctypes.byref(d), None, None, 0, None) == capi.DSPARK_INVALID_ARG
    d.U = 0x10004
    assert capi.dspark_draft_and_schedule(d, s, 0x20000, 1 << 30, 0) == capi.DSPARK_INVALID_ARG  # misaligned U
    d.U = 0x10000
    assert capi.dspark_draft_and_schedule(d, s, 0x20000, 16, 0) == capi.DSPARK_INVALID_ARG  # workspace too small
    s.conf_logit = 0x30000  # not the draft's confidences
    assert capi.dspark_draft_and_schedule(d, s, 0x20000, 1 << 30, 0) == capi.DSPARK_INVALID_ARG
    s.conf_logit, s.gamma = d.conf_logit, 6  # shape differs from the draft's
    assert capi.dspark_draft_and_schedule(d, s, 0x20000, 1 << 30, 0) == capi.DSPARK_INVALID_ARG
    s.gamma, s.mode = 7, 9
    assert capi.dspark_draft_and_schedule(d, s, 0x20000, 1 << 30, 0) == capi.DSPARK_INVALID_ARG
    s.mode = capi.DSPARK_SCHED_GREEDY
    d.dims, s.B = capi.dspark_dims(0, 7, 64, 8, 16, capi.DSPARK_F32), 0
    assert capi.dspark_draft_and_schedule(d, s, 0, 0, 0) == capi.DSPARK_OK  # empty batch

    v = capi.dspark_verify_args()
    v.dims = capi.dspark_dims(4, 4, 64, 0, 0, capi.DSPARK_BF16)
    assert capi.dspark_verify(v, 0, 0, 0) == capi.DSPARK_INVALID_ARG
    v.dims = capi.dspark_dims(0, 4, 64, 0, 0, capi.DSPARK_BF16)
    assert capi.dspark_verify(v, 0, 0, 0) == capi.DSPARK_OK


def test_struct_layouts_match_header(lib):
    # field order and sizes of the ctypes mirrors (64-bit ABI)
    assert ctypes.sizeof(capi.dspark_dims) == 24
    assert capi.dspark_draft_args.seed.offset == 24 + 8 * 8
    assert ctypes.sizeof(capi.dspark_draft_args) == 24 + 8 * 8 + 8 + 5 * 8 + 8 + 8 + 8
    assert ctypes.sizeof(capi.dspark_sched_args) == 16 + 15 * 8
    assert capi.dspark_verify_args.seed.offset == 24 + 8 * 8
    assert ctypes.sizeof(capi.dspark_verify_args) == 24 + 8 * 8 + 8 + 4 * 8 + 8 + 5 * 8


def test_sts_fit_argument_checks(lib):
    st, n = capi.dspark_sts_fit_workspace_size(131072, 7, 128, 15)
    assert st == capi.DSPARK_OK and n >= 7 * 15 * 128 * 12 + 7 * 131072 * 4
    assert capi.dspark_sts_fit_workspace_size(0, 7, 128, 15)[0] == capi.DSPARK_OK
    for bad in [(-1, 7, 128, 15), (10, 0, 128, 15), (10, 33, 128, 15), (10, 7, 0, 15), (10, 7, 128, 0),
                (capi.DSPARK_STS_MAX_SAMPLES + 1, 7, 128, 15), (10, 7, 128, 129), (10, 7, 1024, 17)]:
        assert capi.dspark_sts_fit_workspace_size(*bad)[0] == capi.DSPARK_INVALID_ARG, bad
    assert capi.dspark_sts_fit_workspace_size(10, 7, 1024, 16)[0] == capi.DSPARK_OK
    a = capi.dspark_sts_fit_args()
    a.N, a.gamma, a.n_grid, a.n_bins = 10, 3, 8, 15
    assert capi.dspark_sts_fit(a, 0, 0, 0) == capi.DSPARK_INVALID_ARG  # null pointers
    a.conf_logit = a.accept_len = a.grid = a.sts_temp = a.ece = 256
    assert capi.dspark_sts_fit(a, 0, 0, 0) == capi.DSPARK_INVALID_ARG  # no workspace
    assert capi.dspark_sts_fit(a, 256 + 16, 1 << 20, 0) == capi.DSPARK_INVALID_ARG  # misaligned
    assert capi.dspark_sts_fit(a, 256, 16, 0) == capi.DSPARK_INVALID_ARG  # too small
    a.n_bins = 200
    assert capi.dspark_sts_fit(a, 256, 1 << 20, 0) == capi.DSPARK_INVALID_ARG  # table limit
    assert ctypes.sizeof(capi.dspark_sts_fit_args) == 16 + 6 * 8


def test_pack_rows_argument_checks(lib):
    a = capi.dspark_pack_args()
    a.V, a.dtype, a.rows_per_request, a.max_rows, a.n_src_rows = 64, capi.DSPARK_BF16, 5, 10, 50
    assert capi.dspark_pack_rows(a, 0, 0) == capi.DSPARK_INVALID_ARG  # null pointers
    a.src = a.mark_req = a.mark_pos = a.n_rows = a.dst = 256
    assert capi.dspark_pack_rows(a, 256 + 8, 0) == capi.DSPARK_INVALID_ARG  # misaligned workspace
    for field, bad in [("V", 0), ("dtype", 7), ("rows_per_request", 0), ("max_rows", -1), ("n_src_rows", -1)]:
        b = capi.dspark_pack_args.from_buffer_copy(a)
        setattr(b, field, bad)
        assert capi.dspark_pack_rows(b, 0, 0) == capi.DSPARK_INVALID_ARG, field
    b = capi.dspark_pack_args.from_buffer_copy(a)
    b.max_rows = 0
    assert capi.dspark_pack_rows(b, 0, 0) == capi.DSPARK_OK  # nothing to launch
    assert ctypes.sizeof(capi.dspark_pack_args) == 16 + 8 + 5 * 8


def test_row_free_argument_checks(lib):
    # a draft without p_d rows needs pd_stat (and the Markov head)
    a = capi.dspark_draft_args()
    a.dims = capi.dspark_dims(4, 3, 1024, 64, 8, capi.DSPARK_BF16)
    a.U = a.W1 = a.W2 = a.h = a.w = a.anchor = a.temp = a.req_id = a.tokens = a.pd_tok = 256
    a.conf_logit = a.conf = 256
    assert capi.dspark_draft_sample(a, 256, 1 << 30, 0) == capi.DSPARK_INVALID_ARG  # no rows, no pd_stat
    a.pd_stat, a.head, a.W_rnn = 256, capi.DSPARK_HEAD_RNN, 256
    assert capi.dspark_draft_sample(a, 256, 1 << 30, 0) == capi.DSPARK_INVALID_ARG  # RNN head without rows
    # the rejection residual needs the draft's inputs and pd_stat; any other mode is refused
    v = capi.dspark_verify_args()
    v.dims = capi.dspark_dims(4, 3, 1024, 64, 0, capi.DSPARK_BF16)
    v.target_logits = v.offsets = v.ell = v.tokens = v.pd_tok = v.temp = v.req_id = 256
    v.n_accept = v.out_tok = v.n_out = 256
    assert capi.dspark_verify(v, 256, 1 << 30, 0) == capi.DSPARK_INVALID_ARG  # inverse CDF without rows
    v.residual_mode = capi.DSPARK_RESIDUAL_REJECTION
    assert capi.dspark_verify(v, 256, 1 << 30, 0) == capi.DSPARK_INVALID_ARG  # no U, W1, W2, anchor, pd_stat
    v.residual_mode = 7
    assert capi.dspark_verify(v, 256, 1 << 30, 0) == capi.DSPARK_INVALID_ARG


def _no_visible_gpu():
    # these calls pass made-up device addresses: they must be refused by the
    # argument checks, so they are never made where a GPU could run a kernel
    import torch
    if torch.cuda.is_available():
        pytest.skip("argument-check test with made-up device addresses: CPU only")


def test_misaligned_pointers_are_refused(lib):
    _no_visible_gpu()
    fields = ("U", "W1", "W2", "h", "w", "anchor", "temp", "req_id", "tokens", "pd_rows", "pd_tok", "conf_logit",
              "conf")
    for bad in ("W1", "W2", "h", "w", "pd_rows"):
        a = capi.dspark_draft_args()
        a.dims = capi.dspark_dims(4, 3, 1024, 64, 8, capi.DSPARK_BF16)
        for f in fields:
            setattr(a, f, 0x10000)
        # control: with every address aligned the call passes the checks and
        # fails only at the CUDA layer (no device here)
        assert capi.dspark_draft_sample(a, 0x20000, 1 << 30, 0) == capi.DSPARK_CUDA_ERROR
        setattr(a, bad, 0x10008)
        assert capi.dspark_draft_sample(a, 0x20000, 1 << 30, 0) == capi.DSPARK_INVALID_ARG, bad
    a.pd_rows = 0x10000
    a.head, a.W_rnn = capi.DSPARK_HEAD_RNN, 0x10002
    assert capi.dspark_draft_sample(a, 0x20000, 1 << 30, 0) == capi.DSPARK_INVALID_ARG  # W_rnn
    a.head = 9
    assert capi.dspark_draft_sample(a, 0x20000, 1 << 30, 0) == capi.DSPARK_INVALID_ARG  # unknown head

    for bad in ("target_logits", "pd_rows"):
        v = capi.dspark_verify_args()
        v.dims = capi.dspark_dims(4, 3, 1024, 64, 0, capi.DSPARK_BF16)
        for f in ("target_logits", "offsets", "ell", "tokens", "pd_rows", "pd_tok", "temp", "req_id", "n_accept",
                  "out_tok", "n_out"):
            setattr(v, f, 0x10000)
        assert capi.dspark_verify(v, 0x20000, 1 << 30, 0) == capi.DSPARK_CUDA_ERROR  # control, as above
        setattr(v, bad, 0x10004)
        assert capi.dspark_verify(v, 0x20000, 1 << 30, 0) == capi.DSPARK_INVALID_ARG, bad


def test_noalloc_scheduler_source_names_no_allocating_call():
    # dspark_schedule_noalloc exists for callers that cannot allocate device memory:
    # neither its file nor the scheduler launcher it shares with dspark_schedule
    # may name an allocating runtime call
    csrc = os.path.join(ROOT, "draft_sampling_lossless_markov_gb300", "csrc")
    noalloc = open(os.path.join(csrc, "schedule_noalloc.cu")).read()
    sched = open(os.path.join(csrc, "schedule.cu")).read()
    launcher = sched[sched.index("cudaError_t launch_schedule("):]
    bad = re.compile(r"\b(cudaMalloc\w*|cudaFree\w*|cuMem(?:Alloc|Free|Create|Map)\w*|cudaHostAlloc|cudaMemPool\w*)\b")
    for name, src in (("schedule_noalloc.cu", noalloc), ("launch_schedule", launcher)):
        code = re.sub(r"//[^\n]*", "", src)  # comments may name them
        assert not bad.search(code), (name, bad.search(code).group(0))
