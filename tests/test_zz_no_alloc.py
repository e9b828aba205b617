"""ssd_prefill_varlen_noalloc: the prefill for callers that cannot allocate
device memory at call time (an engine that reserved all free memory for its
state cache, or a host with only the C ABI).  Its scratch is a fixed device
array inside the library.  Called through the C ABI, it must agree with
ssd_prefill_varlen (given caller workspace) and with the oracle on y and on
every stored state, within the parity tolerance, on three calls in a row, each
smaller than the one before -- every later call finds an earlier call's
leftovers in the shared array.  This file is collected last
so that a failure here cannot hide any other test's result."""
import ctypes

import pytest
import torch

import selective_state_space_mamba2_gb300 as ssd
from selective_state_space_mamba2_gb300 import _binding as B
from selective_state_space_mamba2_gb300 import workloads as W
from tests import parity as PT

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _args_for(case, meta, y, err):
    dev = case["x"].device
    t = {k: torch.from_numpy(v).to(dev) for k, v in meta.items()}
    a = ssd.prefill_args(case["x"], case["dt"], case["A"], case["B"], case["C"], case["cu_seqlens"].to(dev),
                         t["cu_chunk_seqlens"], t["seq_idx"], t["last_chunk_indices"], y, t["init_slot"],
                         t["chunk_slot"], case["cache"], case["D"], case["dt_bias"],
                         null_block_id=case["null_block_id"], chunk_size=case["chunk_size"], err_word=err)
    return a, t  # keep the metadata tensors alive with the arguments


def _compare_once(case):
    meta = PT.prefill_metadata(case)
    start = case["cache"].clone()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    # the existing entry point, caller workspace
    y_ref, _ = PT.run_prefill(case, meta=meta, err=err)
    torch.cuda.synchronize()
    cache_ref = case["cache"].clone()
    # the no-allocation entry point on the same inputs and the same starting cache
    case["cache"].copy_(start)
    y = torch.full_like(case["x"], float("nan"))
    a, keep = _args_for(case, meta, y, err)
    rc = ssd.lib().ssd_prefill_varlen_noalloc(ctypes.byref(a),
                                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == B.SSD_OK and int(err.item()) == 0
    tol = PT.TOL[case["x"].dtype]
    e_y = PT.y_err_pair(y.double().cpu().numpy(), y_ref.double().cpu().numpy(), case["x"].dtype)
    written = sorted({int(v) for v in meta["chunk_slot"] if int(v) != case["null_block_id"]})
    w = torch.tensor(written, device=DEV)
    e_s = PT.rel_err(case["cache"][w].double().cpu().numpy(), cache_ref[w].double().cpu().numpy())
    assert e_y <= tol and e_s <= tol, (e_y, e_s, tol)
    others = torch.ones(case["cache"].shape[0], dtype=torch.bool, device=DEV)
    others[w] = False
    assert torch.equal(case["cache"][others].view(torch.int32), start[others].view(torch.int32))
    # and y and every stored state against the oracle directly
    o_y, o_s, o_same, o_tol = PT.check_prefill(case, y, meta, start, case["cache"])
    assert o_y <= o_tol and o_s <= o_tol and o_same, (o_y, o_s, o_same)


def test_noalloc_matches_workspace_entry_point_and_oracle_three_times():
    ssd.build()
    # three different calls in a row, each smaller than the one before, so every scratch byte a
    # later call reads was left there by an earlier one (which must not matter)
    _compare_once(W.prefill_case(32, [2048], [0], 48, 64, 128, 4, 2048, device=DEV, mode="default",
                                 has_init=[False], num_slots=4))
    _compare_once(W.prefill_case(31, [150, 40, 300], [10, 0, 64], 4, 32, 64, 2, 64, dtype=torch.float32,
                                 device=DEV, has_init=[True, False, True], num_slots=40))
    _compare_once(W.prefill_case(34, [70, 33], [5, 0], 2, 16, 32, 1, 32, dtype=torch.float32, device=DEV,
                                 has_init=[True, False], num_slots=12))


def test_noalloc_refuses_calls_beyond_its_scratch():
    ssd.build()
    case = W.prefill_case(33, [8192] * 4, [0] * 4, 48, 64, 128, 4, 256, device=DEV, num_slots=200)
    meta = PT.prefill_metadata(case)
    y = torch.empty_like(case["x"])
    a, keep = _args_for(case, meta, y, None)
    before = case["cache"].clone()
    rc = ssd.lib().ssd_prefill_varlen_noalloc(ctypes.byref(a), None)
    assert rc == B.SSD_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.equal(case["cache"].view(torch.int32), before.view(torch.int32))
