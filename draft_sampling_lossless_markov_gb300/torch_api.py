"""Torch-tensor front end of the C ABI: turns tensors into the C structs.

PyTorch only provides device memory and streams here.  Each function checks
that its tensors are contiguous CUDA tensors of the expected dtype, fills the C
struct with their addresses and calls the library; a non-OK status raises.
Output tensors may be passed in (`out=`) to avoid allocation in a timed loop.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from . import capi


class DsparkError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = f"{fn} returned {capi.dspark_status_string(status)}"
        if status == capi.DSPARK_CUDA_ERROR:
            msg += f" (cudaError {capi.dspark_last_cuda_error()})"
        super().__init__(msg)
        self.status = status


def _check(fn: str, st: int):
    if st != capi.DSPARK_OK:
        raise DsparkError(fn, st)


_DT = {torch.bfloat16: capi.DSPARK_BF16, torch.float32: capi.DSPARK_F32}


def _ptr(t: Optional[torch.Tensor], dtype=None) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("dspark tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("dspark tensors must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def dims(B, gamma, V, r, H, dtype) -> capi.dspark_dims:
    return capi.dspark_dims(int(B), int(gamma), int(V), int(r), int(H), _DT[dtype] if dtype in _DT else int(dtype))


@dataclass
class Workspace:
    buf: torch.Tensor

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()

    @property
    def nbytes(self) -> int:
        return self.buf.numel()

    @classmethod
    def create(cls, d: capi.dspark_dims, device="cuda", stream=None) -> "Workspace":
        st, n = capi.dspark_workspace_size(d)
        _check("dspark_workspace_size", st)
        buf = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
        ws = cls(buf)
        _check("dspark_workspace_init", capi.dspark_workspace_init(ws.ptr, ws.nbytes, _stream(stream)))
        return ws

    def read_error(self, stream=None):
        st, code, detail = capi.dspark_read_error(self.ptr, _stream(stream))
        _check("dspark_read_error", st)
        return code, detail


def _draft_args(U, W1, W2, h, w, anchor, temp, req_id, seed, out, W_rnn, rows, want_pd_stat):
    B, G, V = U.shape
    r = W1.shape[1] if W1 is not None else 0
    H = h.shape[2] if h is not None else 0
    dt = U.dtype
    dev = U.device
    if out is None:
        out = dict(tokens=torch.empty((B, G), dtype=torch.int32, device=dev),
                   pd_tok=torch.empty((B, G), dtype=torch.float32, device=dev),
                   conf_logit=torch.empty((B, G), dtype=torch.float32, device=dev),
                   conf=torch.empty((B, G), dtype=torch.float32, device=dev))
        if rows:
            out["pd_rows"] = torch.empty((B, G, V), dtype=torch.float32, device=dev)
        if want_pd_stat or not rows:
            out["pd_stat"] = torch.empty((B, G, 2), dtype=torch.float32, device=dev)
    a = capi.dspark_draft_args()
    a.dims = dims(B, G, V, r, H, dt)
    a.U, a.W1, a.W2, a.h, a.w = _ptr(U, dt), _ptr(W1, dt), _ptr(W2, dt), _ptr(h, dt), _ptr(w, dt)
    a.anchor, a.temp = _ptr(anchor, torch.int32), _ptr(temp, torch.float32)
    a.req_id = _ptr(req_id, torch.int32)
    a.seed = int(seed)
    a.tokens, a.pd_rows = _ptr(out["tokens"], torch.int32), _ptr(out.get("pd_rows"), torch.float32)
    a.pd_stat = _ptr(out.get("pd_stat"), torch.float32)
    a.pd_tok, a.conf_logit = _ptr(out["pd_tok"], torch.float32), _ptr(out["conf_logit"], torch.float32)
    a.conf = _ptr(out["conf"], torch.float32)
    if W_rnn is not None:
        a.W_rnn, a.head = _ptr(W_rnn, dt), capi.DSPARK_HEAD_RNN
    return a, out


def draft_sample(ws: Workspace, U, W1, W2, h, w, anchor, temp, req_id, seed: int, out: Optional[dict] = None,
                 stream=None, W_rnn=None, rows: bool = True, want_pd_stat: bool = False) -> dict:
    """dspark_draft_sample; W_rnn [3r, 2r + H] (the dtype of U) selects the RNN head;
    rows=False draws without p_d rows (pd_stat [B, gamma, 2] is then returned)."""
    a, out = _draft_args(U, W1, W2, h, w, anchor, temp, req_id, seed, out, W_rnn, rows, want_pd_stat)
    _check("dspark_draft_sample", capi.dspark_draft_sample(a, ws.ptr, ws.nbytes, _stream(stream)))
    return out


def _sched_args(conf_logit, sts_temp, sps, anchor, tokens, mode, out, n_verify_host, want_surv, conf_logit_prev):
    B, G = conf_logit.shape
    dev = conf_logit.device
    cap = B * (1 + G)
    if out is None:
        out = dict(ell=torch.empty(B, dtype=torch.int32, device=dev),
                   offsets=torch.empty(B + 1, dtype=torch.int32, device=dev),
                   flat_tok=torch.empty(cap, dtype=torch.int32, device=dev),
                   mark_req=torch.empty(cap, dtype=torch.int32, device=dev),
                   mark_pos=torch.empty(cap, dtype=torch.int32, device=dev),
                   n_verify=torch.empty(1, dtype=torch.int32, device=dev),
                   theta_best=torch.empty(1, dtype=torch.float64, device=dev))
        if want_surv:
            out["surv"] = torch.empty((B, G), dtype=torch.float32, device=dev)
    if isinstance(sps, np.ndarray):
        sps = torch.from_numpy(np.ascontiguousarray(sps, dtype=np.float64)).to(dev)
    a = capi.dspark_sched_args()
    a.B, a.gamma, a.mode = B, G, int(mode)
    a.conf_logit, a.sts_temp = _ptr(conf_logit, torch.float32), _ptr(sts_temp, torch.float32)
    a.sps = _ptr(sps, torch.float64) if sps is not None else None
    a.anchor, a.tokens = _ptr(anchor, torch.int32), _ptr(tokens, torch.int32)
    a.ell, a.offsets = _ptr(out["ell"], torch.int32), _ptr(out["offsets"], torch.int32)
    a.flat_tok, a.mark_req = _ptr(out["flat_tok"], torch.int32), _ptr(out["mark_req"], torch.int32)
    a.mark_pos, a.n_verify = _ptr(out["mark_pos"], torch.int32), _ptr(out["n_verify"], torch.int32)
    a.theta_best = _ptr(out["theta_best"], torch.float64)
    a.n_verify_host = n_verify_host.data_ptr() if n_verify_host is not None else None
    a.surv = _ptr(out.get("surv"), torch.float32)
    a.conf_logit_prev = _ptr(conf_logit_prev, torch.float32) if conf_logit_prev is not None else None
    out["_sps"] = sps  # keep the table alive while the call is in flight
    return a, out


def schedule(ws: Workspace, conf_logit, sts_temp, sps, anchor, tokens, mode: int, out: Optional[dict] = None,
             stream=None, n_verify_host: Optional[torch.Tensor] = None, want_surv=False,
             conf_logit_prev=None) -> dict:
    a, out = _sched_args(conf_logit, sts_temp, sps, anchor, tokens, mode, out, n_verify_host, want_surv,
                         conf_logit_prev)
    _check("dspark_schedule", capi.dspark_schedule(a, ws.ptr, ws.nbytes, _stream(stream)))
    return out


def draft_and_schedule(ws: Workspace, U, W1, W2, h, w, anchor, temp, req_id, seed: int, sts_temp, sps, mode: int,
                       out: Optional[dict] = None, sched_out: Optional[dict] = None, stream=None, W_rnn=None,
                       rows: bool = True, want_pd_stat: bool = False, n_verify_host: Optional[torch.Tensor] = None,
                       want_surv=False, conf_logit_prev=None) -> tuple:
    """dspark_draft_and_schedule: draft_sample then schedule of its confidences
    and tokens, in one call that may overlap them; returns (draft out, schedule out)."""
    da, out = _draft_args(U, W1, W2, h, w, anchor, temp, req_id, seed, out, W_rnn, rows, want_pd_stat)
    sa, sched_out = _sched_args(out["conf_logit"], sts_temp, sps, anchor, out["tokens"], mode, sched_out,
                                n_verify_host, want_surv, conf_logit_prev)
    _check("dspark_draft_and_schedule",
           capi.dspark_draft_and_schedule(da, sa, ws.ptr, ws.nbytes, _stream(stream)))
    return out, sched_out


def verify(ws: Workspace, target_logits, offsets, ell, tokens, pd_rows, pd_tok, temp, req_id, seed: int,
           out: Optional[dict] = None, stream=None, commit_cap=None, rejection: Optional[dict] = None) -> dict:
    """dspark_verify; commit_cap [B] i32 (the scheduled windows) selects cap-accept;
    rejection=dict(U, W1, W2, anchor, pd_stat) draws the residual by rejection
    from p_t (pd_rows may then be None)."""
    B, G = tokens.shape
    V = target_logits.shape[-1]
    dev = tokens.device
    dt = target_logits.dtype
    if out is None:
        out = dict(n_accept=torch.empty(B, dtype=torch.int32, device=dev),
                   out_tok=torch.empty((B, G + 1), dtype=torch.int32, device=dev),
                   n_out=torch.empty(B, dtype=torch.int32, device=dev))
    a = capi.dspark_verify_args()
    a.dims = dims(B, G, V, rejection["W1"].shape[1] if rejection else 0, 0, dt)
    a.target_logits = _ptr(target_logits, dt)
    a.offsets, a.ell, a.tokens = _ptr(offsets, torch.int32), _ptr(ell, torch.int32), _ptr(tokens, torch.int32)
    a.pd_rows, a.pd_tok = _ptr(pd_rows, torch.float32), _ptr(pd_tok, torch.float32)
    a.temp, a.req_id = _ptr(temp, torch.float32), _ptr(req_id, torch.int32)
    if rejection is not None:
        a.residual_mode = capi.DSPARK_RESIDUAL_REJECTION
        a.U, a.W1, a.W2 = _ptr(rejection["U"], dt), _ptr(rejection["W1"], dt), _ptr(rejection["W2"], dt)
        a.anchor, a.pd_stat = _ptr(rejection["anchor"], torch.int32), _ptr(rejection["pd_stat"], torch.float32)
    a.seed = int(seed)
    a.n_accept, a.out_tok, a.n_out = (_ptr(out["n_accept"], torch.int32), _ptr(out["out_tok"], torch.int32),
                                      _ptr(out["n_out"], torch.int32))
    a.commit_cap = _ptr(commit_cap, torch.int32) if commit_cap is not None else None
    _check("dspark_verify", capi.dspark_verify(a, ws.ptr, ws.nbytes, _stream(stream)))
    return out


def sts_fit_workspace(N: int, gamma: int, n_grid: int, n_bins: int, device="cuda", stream=None) -> Workspace:
    """Workspace of dspark_sts_fit (separate from the step workspace)."""
    st, n = capi.dspark_sts_fit_workspace_size(int(N), int(gamma), int(n_grid), int(n_bins))
    _check("dspark_sts_fit_workspace_size", st)
    ws = Workspace(torch.empty(max(n, 256), dtype=torch.uint8, device=device))
    _check("dspark_workspace_init", capi.dspark_workspace_init(ws.ptr, ws.nbytes, _stream(stream)))
    return ws


def sts_fit(ws: Workspace, conf_logit, accept_len, grid, n_bins: int, out: Optional[dict] = None, stream=None):
    """dspark_sts_fit: conf_logit [N, gamma] f32, accept_len [N] i32, grid [G] f32.
    Returns dict(sts_temp [gamma] f32, grid_index [gamma] i32, ece [gamma, G] f64)."""
    N, G = conf_logit.shape
    n_grid = grid.numel()
    dev = conf_logit.device
    if out is None:
        out = dict(sts_temp=torch.empty(G, dtype=torch.float32, device=dev),
                   grid_index=torch.empty(G, dtype=torch.int32, device=dev),
                   ece=torch.empty((G, n_grid), dtype=torch.float64, device=dev))
    a = capi.dspark_sts_fit_args()
    a.N, a.gamma, a.n_grid, a.n_bins = int(N), int(G), int(n_grid), int(n_bins)
    a.conf_logit = _ptr(conf_logit, torch.float32)
    a.accept_len = _ptr(accept_len, torch.int32)
    a.grid = _ptr(grid, torch.float32)
    a.sts_temp = _ptr(out["sts_temp"], torch.float32)
    a.grid_index = _ptr(out.get("grid_index"), torch.int32)
    a.ece = _ptr(out["ece"], torch.float64)
    _check("dspark_sts_fit", capi.dspark_sts_fit(a, ws.ptr, ws.nbytes, _stream(stream)))
    return out


def pack_rows(src, mark_req, mark_pos, n_rows, dst, ws: Optional[Workspace] = None, stream=None):
    """dspark_pack_rows: dst[i] = src[mark_req[i], mark_pos[i]] for i < n_rows[0].

    src [R, rows_per_request, V]: a CUDA tensor or a pinned CPU tensor (read by
    the GPU in place); mark_req, mark_pos [max_rows] and n_rows [1] int32 CUDA
    tensors; dst [max_rows, V] CUDA tensor of src's dtype."""
    if not src.is_contiguous() or not (src.is_cuda or src.is_pinned()):
        raise ValueError("src must be a contiguous CUDA tensor or a pinned CPU tensor")
    if src.dtype != dst.dtype:
        raise TypeError("src and dst dtypes differ")
    R, G1, V = src.shape
    a = capi.dspark_pack_args()
    a.V, a.dtype, a.rows_per_request, a.max_rows = int(V), _DT[src.dtype], int(G1), int(dst.shape[0])
    a.n_src_rows = int(R * G1)
    a.src = src.data_ptr()
    a.mark_req, a.mark_pos = _ptr(mark_req, torch.int32), _ptr(mark_pos, torch.int32)
    a.n_rows, a.dst = _ptr(n_rows, torch.int32), _ptr(dst)
    _check("dspark_pack_rows", capi.dspark_pack_rows(a, ws.ptr if ws is not None else 0, _stream(stream)))
    return dst
