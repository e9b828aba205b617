"""ssd_mixed_step (the prefill part and the decode part of one step, issued together) against
the fp64 oracle, and bit for bit against the two calls made one after the other."""
import ctypes
import math

import numpy as np
import pytest
import torch

import selective_state_space_mamba2_gb300 as ssd
from selective_state_space_mamba2_gb300 import workloads as W
from tests import parity as PT

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    ssd.build()
    torch.cuda.init()


def _case(num_prefills, prefill_len, P, num_decodes, seed):
    H, G, N, Q = 8, 2, 128, 256
    cols = (prefill_len + Q - 1) // Q
    pre, dec = W.long_mixed(device=DEV, seed=seed, num_prefills=num_prefills, prefill_len=prefill_len,
                            num_decodes=num_decodes, chunk_size=Q, H=H, P=P, N=N, G=G,
                            num_slots=num_prefills * cols + num_decodes + 8)
    return pre, dec


def _pargs(pre, meta, y, err):
    t = {k: torch.from_numpy(v).to(DEV) for k, v in meta.items()}
    t["cu_seqlens"] = pre["cu_seqlens"].to(DEV)  # kept alive with the rest: the args hold raw pointers
    pa = ssd.prefill_args(pre["x"], pre["dt"], pre["A"], pre["B"], pre["C"], t["cu_seqlens"],
                          t["cu_chunk_seqlens"], t["seq_idx"], t["last_chunk_indices"], y, t["init_slot"],
                          t["chunk_slot"], pre["cache"], pre["D"], pre["dt_bias"],
                          null_block_id=pre["null_block_id"], chunk_size=pre["chunk_size"], err_word=err,
                          seq_order=t.get("seq_order"))
    return pa, t


def _args(pre, dec, meta, y, yd, err):
    pa, t = _pargs(pre, meta, y, err)
    si = dec["state_indices"].to(DEV)
    da = ssd.decode_args(dec["x"], dec["dt"], dec["A"], dec["B"], dec["C"], dec["cache"], si, yd, D=dec["D"],
                         dt_bias=dec["dt_bias"], null_block_id=dec["null_block_id"], err_word=err)
    return pa, da, (t, si)  # the device metadata stays alive with the argument sets


@pytest.mark.parametrize("num_prefills,prefill_len,P", [
    (3, 900, 64),   # tensor-core path, one CTA per (sequence, head), ragged last block
    (1, 2048, 64),  # tensor-core path with the segment pass (one sequence cut into segments)
    (2, 500, 32),   # headdim 32: the CUDA-core prefill, the decode started at once
])
def test_mixed_step_matches_the_oracle_and_the_two_calls(num_prefills, prefill_len, P):
    pre, dec = _case(num_prefills, prefill_len, P, num_decodes=24, seed=60 + P + num_prefills)
    cache = pre["cache"]
    assert dec["cache"] is cache  # one cache, slots distinct across the two parts
    before = cache.clone()
    meta = PT.prefill_metadata(pre)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = torch.full_like(pre["x"], float("nan"))
    yd = torch.full_like(dec["x"], float("nan"))
    pa, da, keep = _args(pre, dec, meta, y, yd, err)
    ssd.ssd_mixed_step(pa, da)
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    e_y, e_s, _, tol = PT.check_prefill(pre, y, meta, before, cache)
    assert e_y <= tol and e_s <= tol, (e_y, e_s)
    e_yd, e_sd, dead_ok, tol_d, nlive = PT.check_decode(dec, yd, before, cache, check_untouched=False)
    assert nlive == 24 and dead_ok and e_yd <= tol_d and e_sd <= tol_d, (e_yd, e_sd)
    written = {int(s) for s in meta["chunk_slot"] if int(s) != pre["null_block_id"]}
    written |= {int(s) for s in dec["state_indices"].flatten().tolist()}
    mask = torch.ones(cache.shape[0], dtype=torch.bool, device=DEV)
    mask[torch.tensor(sorted(written), device=DEV)] = False
    assert torch.equal(cache[mask].view(torch.int32), before[mask].view(torch.int32))

    # the same two calls one after the other, from the same cache: the same bits
    got = (y.clone(), yd.clone(), cache.clone())
    cache.copy_(before)
    y.fill_(float("nan"))
    yd.fill_(float("nan"))
    assert ssd.lib().ssd_prefill_varlen(ctypes.byref(pa), ctypes.c_void_p(_ws(pa).data_ptr()),
                                        _ws(pa).numel(), None) == 0
    assert ssd.lib().ssm_decode_update(ctypes.byref(da), None) == 0
    torch.cuda.synchronize()
    assert torch.equal(got[0].view(torch.int16), y.view(torch.int16))
    assert torch.equal(got[1].view(torch.int16), yd.view(torch.int16))
    assert torch.equal(got[2].view(torch.int32), cache.view(torch.int32))
    del keep


_WS = {}


def _ws(pa):
    n = max(ssd.ssd_prefill_workspace_size(pa), 1)
    if _WS.get("n", 0) < n:
        _WS["t"] = torch.empty(n, dtype=torch.uint8, device=DEV)
        _WS["n"] = n
    return _WS["t"]


def test_mixed_step_with_one_part_empty_is_the_other_call():
    pre, dec = _case(2, 640, 64, num_decodes=8, seed=71)
    cache = pre["cache"]
    before = cache.clone()
    meta = PT.prefill_metadata(pre)
    y = torch.full_like(pre["x"], float("nan"))
    yd = torch.full_like(dec["x"], float("nan"))
    pa, da, keep = _args(pre, dec, meta, y, yd, None)
    empty_d = ssd.decode_args(dec["x"], dec["dt"], dec["A"], dec["B"], dec["C"], dec["cache"], keep[1], yd,
                              D=dec["D"], dt_bias=dec["dt_bias"], null_block_id=dec["null_block_id"])
    empty_d.batch = 0
    ssd.ssd_mixed_step(pa, empty_d)
    torch.cuda.synchronize()
    assert torch.isnan(yd).all()  # nothing of the decode ran
    e_y, e_s, _, tol = PT.check_prefill(pre, y, meta, before, cache)
    assert e_y <= tol and e_s <= tol and not math.isnan(e_y)
    cache.copy_(before)
    y.fill_(float("nan"))
    empty_p = ssd.prefill_args(pre["x"], pre["dt"], pre["A"], pre["B"], pre["C"], keep[0]["cu_seqlens"],
                               keep[0]["cu_chunk_seqlens"], keep[0]["seq_idx"], keep[0]["last_chunk_indices"], y,
                               keep[0]["init_slot"], keep[0]["chunk_slot"], pre["cache"], pre["D"],
                               pre["dt_bias"], null_block_id=pre["null_block_id"], chunk_size=pre["chunk_size"])
    empty_p.total_tokens, empty_p.num_chunks = 0, 0
    ssd.ssd_mixed_step(empty_p, da)
    torch.cuda.synchronize()
    assert torch.isnan(y).all()  # nothing of the prefill ran
    e_yd, e_sd, dead_ok, tol_d, nlive = PT.check_decode(dec, yd, before, cache)
    assert nlive == 8 and dead_ok and e_yd <= tol_d and e_sd <= tol_d, (e_yd, e_sd)


@pytest.mark.parametrize("P,tpr", [(64, 1), (64, 3), (32, 4), (16, 2), (8, 9)])
def test_decode_beside_a_tensor_core_prefill(P, tpr):
    """A decode part of another headdim than the prefill's, with speculative columns (more tokens
    than one staging batch in the last case) and its own cache, against the oracle."""
    pre, _ = _case(2, 700, 64, num_decodes=1, seed=80 + P + tpr)
    dec = W.decode_case(90 + P + tpr, live=11, padded=16, tokens_per_req=tpr, H=8, P=P, N=128, G=2,
                        num_slots=200, device=DEV)
    if tpr > 1:  # one live request skips a write (not the column it reads from)
        dec["state_indices"][3, (int(dec["num_accepted"][3]) + 1) % tpr] = dec["null_block_id"]
    before_p, before_d = pre["cache"].clone(), dec["cache"].clone()
    meta = PT.prefill_metadata(pre)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = torch.full_like(pre["x"], float("nan"))
    yd = torch.full_like(dec["x"], float("nan"))
    pa, keep = _pargs(pre, meta, y, err)
    na = dec["num_accepted"].to(DEV)
    si = dec["state_indices"].to(DEV)
    da = ssd.decode_args(dec["x"], dec["dt"], dec["A"], dec["B"], dec["C"], dec["cache"], si, yd, na, D=dec["D"],
                         dt_bias=dec["dt_bias"], null_block_id=dec["null_block_id"], err_word=err)
    ssd.ssd_mixed_step(pa, da)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    e_y, e_s, same_p, tol = PT.check_prefill(pre, y, meta, before_p, pre["cache"])
    assert e_y <= tol and e_s <= tol and same_p, (e_y, e_s)
    e_yd, e_sd, ok, tol_d, nlive = PT.check_decode(dec, yd, before_d, dec["cache"])
    assert nlive == 11 and ok and e_yd <= tol_d and e_sd <= tol_d, (e_yd, e_sd)
    del keep, na, si


def test_long_mixed_step_full_size_sampled():
    """The benchmark's step at full size, in the configuration it is timed in (one ssd_mixed_step
    call): 8 x 65536 prefill tokens and 384 decodes on a 16384-slot cache.  y and all 2048 chunk
    states on two heads, six decode requests in full, fingerprints of every slot neither part
    writes."""
    pre, dec = W.long_mixed(DEV)
    cache = pre["cache"]
    reqs = [0, 1, 77, 200, 301, 383]
    read_before = {int(dec["state_indices"][r, 0]): cache[int(dec["state_indices"][r, 0])].clone() for r in reqs}
    fp_before = PT.slot_fingerprints(cache)
    meta = PT.prefill_metadata(pre)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = torch.empty_like(pre["x"])
    yd = torch.full_like(dec["x"], float("nan"))
    pa, da, keep = _args(pre, dec, meta, y, yd, err)
    ssd.ssd_mixed_step(pa, da)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    heads = [3, 126]
    yo, cso = PT.oracle_prefill(pre, meta, cache, heads=heads)
    hs = torch.tensor(heads)
    tol = PT.TOL[torch.bfloat16]
    assert PT.y_err(y[:, hs].double().cpu().numpy(), yo, torch.bfloat16) <= tol
    sl = torch.from_numpy(meta["chunk_slot"].astype(np.int64)).to(DEV)
    assert PT.rel_err(cache[sl][:, hs].double().cpu().numpy(), cso) <= tol
    e_yd, e_sd, _, tol_d, nlive = PT.check_decode(dec, yd, read_before, cache, requests=reqs, check_untouched=False)
    assert nlive == len(reqs) and e_yd <= tol_d and e_sd <= tol_d, (e_yd, e_sd)
    assert not torch.isnan(yd).any()  # every decode row written
    fp_after = PT.slot_fingerprints(cache)
    mask = torch.ones_like(fp_after, dtype=torch.bool)
    mask[sl] = False
    mask[dec["state_indices"][:, 0].long().to(DEV)] = False
    assert torch.equal(fp_after[mask], fp_before[mask])
    del keep


def test_mixed_step_replays_as_a_graph():
    """Captured once (after an eager call has made the library's streams and events) and replayed
    with new token contents and states, the step gives the bits of an eager call on the same
    inputs: the fork onto the library's streams and the join back are captured with it."""
    pre, dec = _case(3, 900, 64, num_decodes=24, seed=91)
    cache = pre["cache"]
    meta = PT.prefill_metadata(pre)
    y = torch.full_like(pre["x"], float("nan"))
    yd = torch.full_like(dec["x"], float("nan"))
    pa, da, keep = _args(pre, dec, meta, y, yd, None)
    ws = torch.empty(max(ssd.ssd_prefill_workspace_size(pa), 1), dtype=torch.uint8, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ssd.ssd_mixed_step(pa, da, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ssd.ssd_mixed_step(pa, da, workspace=ws)
    g = torch.Generator(device=DEV).manual_seed(92)
    for _ in range(2):
        for t in (pre["x"], pre["B"], pre["C"], dec["x"], dec["B"], dec["C"]):
            t.copy_(torch.randn(t.shape, generator=g, device=DEV).to(t.dtype))
        before = cache.clone()
        y.fill_(float("nan"))
        yd.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        got = (y.clone(), yd.clone(), cache.clone())
        cache.copy_(before)
        y.fill_(float("nan"))
        yd.fill_(float("nan"))
        ssd.ssd_mixed_step(pa, da, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(got[0].view(torch.int16), y.view(torch.int16))
        assert torch.equal(got[1].view(torch.int16), yd.view(torch.int16))
        assert torch.equal(got[2].view(torch.int32), cache.view(torch.int32))
        assert not torch.isnan(y).any() and not torch.isnan(yd).any()
    del keep


@pytest.mark.parametrize("P", [64, 32])
def test_mixed_step_with_the_output_gate(P):
    """Both parts gated (y * silu(z)): the tensor-core prefill's gated instance (headdim 64) or the
    CUDA-core one (headdim 32), and the decode's."""
    pre, dec = _case(2, 600, P, num_decodes=12, seed=95 + P)
    g = torch.Generator(device=DEV).manual_seed(96)
    zp = torch.randn(pre["x"].shape, generator=g, device=DEV).to(pre["x"].dtype)
    zd = torch.randn(dec["x"].shape, generator=g, device=DEV).to(dec["x"].dtype)
    cache = pre["cache"]
    before = cache.clone()
    meta = PT.prefill_metadata(pre)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = torch.full_like(pre["x"], float("nan"))
    yd = torch.full_like(dec["x"], float("nan"))
    t = {k: torch.from_numpy(v).to(DEV) for k, v in meta.items()}
    t["cu_seqlens"] = pre["cu_seqlens"].to(DEV)
    pa = ssd.prefill_args(pre["x"], pre["dt"], pre["A"], pre["B"], pre["C"], t["cu_seqlens"], t["cu_chunk_seqlens"],
                          t["seq_idx"], t["last_chunk_indices"], y, t["init_slot"], t["chunk_slot"], cache, pre["D"],
                          pre["dt_bias"], z=zp, null_block_id=pre["null_block_id"], chunk_size=pre["chunk_size"],
                          err_word=err, seq_order=t.get("seq_order"))
    si = dec["state_indices"].to(DEV)
    da = ssd.decode_args(dec["x"], dec["dt"], dec["A"], dec["B"], dec["C"], cache, si, yd, D=dec["D"],
                         dt_bias=dec["dt_bias"], z=zd, null_block_id=dec["null_block_id"], err_word=err)
    ssd.ssd_mixed_step(pa, da)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    e_y, e_s, _, tol = PT.check_prefill(pre, y, meta, before, cache, z=zp)
    assert e_y <= tol and e_s <= tol, (e_y, e_s)
    e_yd, e_sd, ok, tol_d, nlive = PT.check_decode(dec, yd, before, cache, check_untouched=False, z=zd)
    assert nlive == 12 and ok and e_yd <= tol_d and e_sd <= tol_d, (e_yd, e_sd)
    del t, si
