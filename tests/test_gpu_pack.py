"""GPU parity of dspark_pack_rows (the marker gather of the verify batch) against
the oracle's definition, from device memory and from pinned host memory."""
import numpy as np
import pytest
import torch

import synth
from oracle import schedule as S
from gpu_common import check_no_error, require_gpu, to_dev_i32, workspace_for
from draft_sampling_lossless_markov_gb300 import capi
from draft_sampling_lossless_markov_gb300 import torch_api as T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _markers(B, G, seed):
    rng = np.random.default_rng(seed)
    ell = rng.integers(0, G + 1, B)
    fl = S.flatten(ell, np.zeros(B, np.int64), np.zeros((B, G), np.int64))
    cap = B * (G + 1)
    req = np.full(cap, -1, np.int32)
    pos = np.full(cap, -1, np.int32)
    n = int(fl["offsets"][-1])
    req[:n], pos[:n] = fl["mark_req"], fl["mark_pos"]
    return req, pos, n


@pytest.mark.parametrize("B,G,V,dt,where", [
    (7, 3, 1024, torch.bfloat16, "device"),
    (7, 3, 1024, torch.bfloat16, "host"),
    (33, 5, 1001, torch.bfloat16, "device"),   # rows not a multiple of 16 bytes: element path
    (20, 4, 515, torch.float32, "host"),
    (64, 7, 4096, torch.float32, "device"),
])
def test_pack_rows_matches_the_marker_gather(B, G, V, dt, where):
    g = torch.Generator().manual_seed(3)
    src = torch.randn((B, G + 1, V), generator=g).to(dt)
    src = src.pin_memory() if where == "host" else src.cuda()
    req, pos, n = _markers(B, G, B + V)
    dst = torch.full((B * (G + 1), V), -7.0, dtype=dt, device="cuda")
    ws = workspace_for(B, G, V, 0, 0, dt)
    T.pack_rows(src, to_dev_i32(req), to_dev_i32(pos), to_dev_i32([n]), dst, ws)
    torch.cuda.synchronize()
    check_no_error(ws)
    expect = S.pack_rows(src.float().cpu().numpy(), req, pos, n)
    np.testing.assert_array_equal(dst[:n].float().cpu().numpy(), expect)
    assert bool((dst[n:] == -7.0).all())  # rows past the count are not written


def test_pack_rows_unaligned_source_and_bad_marker():
    B, G, V = 5, 2, 64
    base = torch.randn(B * (G + 1) * V + 1, dtype=torch.bfloat16, device="cuda")
    src = base[1:].view(B, G + 1, V)  # 2-byte offset: the element path
    req, pos, n = _markers(B, G, 1)
    req[2] = B + 3  # outside the source
    dst = torch.zeros((B * (G + 1), V), dtype=torch.bfloat16, device="cuda")
    ws = workspace_for(B, G, V, 0, 0, torch.bfloat16)
    T.pack_rows(src, to_dev_i32(req), to_dev_i32(pos), to_dev_i32([n]), dst, ws)
    torch.cuda.synchronize()
    assert ws.read_error() == (capi.DSPARK_BAD_INPUT, 2)
    keep = [i for i in range(n) if i != 2]
    expect = S.pack_rows(src.float().cpu().numpy(), np.where(req < B, req, 0), pos, n)
    np.testing.assert_array_equal(dst[keep].float().cpu().numpy(), expect[keep])
    assert bool((dst[2] == 0).all())


def test_pack_rows_full_size_from_pinned_host():
    # the headline batch: every request's gamma + 1 target rows on the host, the
    # scheduler's markers on the device
    wl = synth.get_workload("sweep_B256_g7")
    B, G, V = wl.B, wl.gamma, wl.V
    g = torch.Generator().manual_seed(5)
    src = torch.randn((B, G + 1, V), generator=g).to(torch.bfloat16).pin_memory()
    req, pos, n = _markers(B, G, 9)
    dst = torch.empty((B * (G + 1), V), dtype=torch.bfloat16, device="cuda")
    T.pack_rows(src, to_dev_i32(req), to_dev_i32(pos), to_dev_i32([n]), dst)
    torch.cuda.synchronize()
    idx = torch.from_numpy(req[:n].astype(np.int64) * (G + 1) + pos[:n])
    assert torch.equal(dst[:n].cpu(), src.view(-1, V).index_select(0, idx))


def test_pack_rows_empty_count_and_empty_launch():
    B, G, V = 4, 2, 64
    src = torch.randn((B, G + 1, V), dtype=torch.bfloat16, device="cuda")
    req, pos, n = _markers(B, G, 2)
    dst = torch.full((B * (G + 1), V), 3.0, dtype=torch.bfloat16, device="cuda")
    T.pack_rows(src, to_dev_i32(req), to_dev_i32(pos), to_dev_i32([0]), dst)  # a count of zero
    torch.cuda.synchronize()
    assert bool((dst == 3.0).all())
    empty = torch.empty((0, V), dtype=torch.bfloat16, device="cuda")
    T.pack_rows(src, to_dev_i32(req), to_dev_i32(pos), to_dev_i32([n]), empty)  # max_rows = 0: no launch
    torch.cuda.synchronize()
