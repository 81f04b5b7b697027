"""Fixtures shared by the GPU tests: build + load the library, run the three calls."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from draft_sampling_lossless_markov_gb300 import build, capi
from draft_sampling_lossless_markov_gb300 import torch_api as T


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    capi.load()


def workspace_for(B, G, V, r, H, dtype) -> T.Workspace:
    return T.Workspace.create(T.dims(B, G, V, r, H, dtype))


def gpu_draft(inp: dict, ws: T.Workspace | None = None) -> tuple[dict, T.Workspace]:
    U = inp["U"]
    B, G, V = U.shape
    r = inp["W1"].shape[1]
    H = inp["h"].shape[2]
    if ws is None:
        ws = workspace_for(B, G, V, r, H, U.dtype)
    out = T.draft_sample(ws, U, inp["W1"] if r else None, inp["W2"] if r else None, inp["h"] if H else None,
                         inp["w"] if H + r else None, inp["anchor"], inp["temp"], inp["req_id"], inp["seed"])
    torch.cuda.synchronize()
    return out, ws


def gather_target_rows(target: torch.Tensor, mark_req: torch.Tensor, mark_pos: torch.Tensor, n: int) -> torch.Tensor:
    """Stand-in for the target model's forward on the flattened batch: the
    synthetic target row of (request, position) for every kept row."""
    G1 = target.shape[1]
    idx = (mark_req[:n].long() * G1 + mark_pos[:n].long())
    return target.reshape(-1, target.shape[2]).index_select(0, idx).contiguous()


def check_no_error(ws: T.Workspace):
    code, detail = ws.read_error()
    assert code == 0, (capi.dspark_status_string(code), detail)


def flatten_np(ell, anchor, tokens):
    from oracle.schedule import flatten
    return flatten(ell, anchor, tokens)


def to_dev_i32(a, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def to_dev_f32(a, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)
