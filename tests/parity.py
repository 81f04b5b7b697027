"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI,
run the fp64 oracle on the same inputs, compare under the tolerance contract.

Tolerance contract:
* greedy tokens, accept counts, verify lengths, offsets and marker tensors are
  compared bit for bit;
* a sampled token must match unless the oracle's fp64 CDF margin at that draw
  is below 1e-5; an accept decision must match unless its relative margin
  |u p_d - p_t| / max(u p_d, p_t) is below 1e-5; a draft-greedy argmax must
  match unless its top-2 logit gap is below 1e-5 max(1, |l_max|); a Theta
  comparison must match unless |Theta_i - Theta_{i-1}| <= 1e-12 Theta_i;
* once a request meets an exempted decision its later outputs are not
  compared (they depend on a legitimately different draw); the count of such
  requests is returned so a test can bound it;
* probabilities and confidences agree within 2e-3 relative for bf16 inputs and
  1e-5 for fp32 inputs (plus 1e-30 absolute for values near fp32 underflow).
"""
from __future__ import annotations

import numpy as np
import torch

MARGIN = 1e-5
THETA_MARGIN = 1e-12


def rtol_for(dtype) -> float:
    return 2e-3 if dtype in (torch.bfloat16, "bf16") else 1e-5


def to_np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def assert_close_rel(gpu, orc, rtol, what, atol=1e-30):
    gpu = np.asarray(gpu, np.float64)
    orc = np.asarray(orc, np.float64)
    bad = np.abs(gpu - orc) > rtol * np.abs(orc) + atol
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} / {bad.size} outside rtol {rtol}; first at {tuple(i)}: "
                             f"gpu {gpu[tuple(i)]!r} oracle {orc[tuple(i)]!r}")


def compare_draft(g: dict, o: dict, rtol: float, check_pd_rows=True) -> dict:
    """g: GPU outputs as numpy (tokens, pd_rows, pd_tok, conf_logit, conf) for the
    same requests, in the same order, as the oracle dict o."""
    R, G = o["tokens"].shape
    exempt = o["margin"] < MARGIN
    first = np.where(exempt.any(axis=1), exempt.argmax(axis=1), G)  # first exempted position per request
    n_tok = 0
    for r in range(R):
        e = first[r]
        # values of position k depend on the tokens before k: compare k <= e
        kk = slice(0, min(e + 1, G))
        zl_o = o["conf_logit"][r, kk]
        if np.any(np.abs(g["conf_logit"][r, kk] - zl_o) > rtol * np.maximum(np.abs(zl_o), 1.0)):
            raise AssertionError(f"conf_logit mismatch request {r}: {g['conf_logit'][r, kk]} vs {zl_o}")
        assert_close_rel(g["conf"][r, kk], o["conf"][r, kk], rtol, f"conf r={r}")
        if check_pd_rows and o.get("pd") is not None:
            assert_close_rel(g["pd_rows"][r, kk], o["pd"][r, kk], rtol, f"pd_rows r={r}")
        # tokens and p_d(x_k) for k < e
        if e > 0:
            np.testing.assert_array_equal(g["tokens"][r, :e], o["tokens"][r, :e], err_msg=f"tokens r={r}")
            assert_close_rel(g["pd_tok"][r, :e], o["pd_tok"][r, :e], rtol, f"pd_tok r={r}")
            n_tok += e
    return dict(n_requests=R, n_exempt_requests=int((first < G).sum()), n_tokens_compared=n_tok)


def compare_schedule(g: dict, o: dict, surv_equal: bool = False) -> bool:
    """Bit-exact comparison of the scheduler's integer outputs; returns False (and
    compares nothing) when the oracle reports an exempted decision.  A calibrated
    confidence whose fp64 sigmoid lies within 1e-13 (relative) of an fp32 rounding
    midpoint is such a decision, unless the caller has already checked that both
    sides produced the same fp32 survival products (surv_equal)."""
    if o["theta_margin"] <= THETA_MARGIN or (not surv_equal and o["sts_margin"] <= 1e-13):
        return False
    R = len(o["ell"])
    N = int(o["offsets"][-1])
    np.testing.assert_array_equal(g["ell"], o["ell"], err_msg="ell")
    np.testing.assert_array_equal(g["offsets"], o["offsets"], err_msg="offsets")
    assert int(g["n_verify"][0]) == N
    np.testing.assert_array_equal(g["flat_tok"][:N], o["flat_tok"], err_msg="flat_tok")
    np.testing.assert_array_equal(g["mark_req"][:N], o["mark_req"], err_msg="mark_req")
    np.testing.assert_array_equal(g["mark_pos"][:N], o["mark_pos"], err_msg="mark_pos")
    assert np.all(g["flat_tok"][N:] == -1) and np.all(g["mark_req"][N:] == -1)
    if o["theta_best"] != 0.0:
        assert abs(g["theta_best"][0] - o["theta_best"]) <= 1e-12 * abs(o["theta_best"]), \
            (g["theta_best"][0], o["theta_best"])
    else:
        assert g["theta_best"][0] == 0.0
    return True


def compare_verify(g: dict, o: dict, greedy: np.ndarray) -> dict:
    """Compare verify outputs request by request; exempted requests are skipped."""
    R = len(o["n_accept"])
    exempt = (o["accept_margin"] < MARGIN) | (o["sample_margin"] < MARGIN)
    exempt &= ~greedy
    for r in range(R):
        if exempt[r]:
            continue
        assert g["n_accept"][r] == o["n_accept"][r], (r, g["n_accept"][r], o["n_accept"][r])
        assert g["n_out"][r] == o["n_out"][r]
        np.testing.assert_array_equal(g["out_tok"][r], o["out_tok"][r], err_msg=f"out_tok r={r}")
    return dict(n_requests=R, n_exempt=int(exempt.sum()))


def np_inputs(inp: dict, idx=None) -> dict:
    """numpy views of the draft inputs (optionally a subset of requests) for the oracle."""
    sel = (lambda t: t[idx]) if idx is not None else (lambda t: t)
    return dict(U=to_np64(sel(inp["U"])), W1=to_np64(inp["W1"]), W2=to_np64(inp["W2"]),
                h=to_np64(sel(inp["h"])), w=to_np64(inp["w"]),
                anchor=sel(inp["anchor"]).cpu().numpy().astype(np.int64),
                temp=sel(inp["temp"]).cpu().numpy().astype(np.float64),
                seed=inp["seed"], req_id=sel(inp["req_id"]).cpu().numpy().astype(np.int64))


def gpu_np(d: dict) -> dict:
    out = {}
    for k, v in d.items():
        if isinstance(v, torch.Tensor):
            out[k] = v.cpu().numpy() if v.dtype != torch.bfloat16 else v.float().cpu().numpy()
    return out
