"""Parity of ssd_prefill_varlen (CUDA, via the C ABI) with the fp64 oracle."""
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


def _err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _run_and_check(case, heads=None, **kw):
    before = case["cache"].clone()
    err = _err()
    y, meta = PT.run_prefill(case, err=err, **kw)
    torch.cuda.synchronize()
    okw = {k: kw[k] for k in ("D", "dt_bias", "dt_limit", "dt_softplus", "z") if k in kw}
    e_y, e_s, same, tol = PT.check_prefill(case, y, meta, before, case["cache"], heads=heads, **okw)
    assert int(err.item()) == 0
    assert e_y <= tol, ("y", e_y, tol)
    assert e_s <= tol, ("state", e_s, tol)
    assert same, "a slot no chunk writes was modified"
    return e_y, e_s


def test_tiny_fp32_single_sequence():
    """1 x 256 tokens, H=4, P=N=16, chunk 64, fp32, zero initial state."""
    _run_and_check(W.tiny_fp32_prefill(DEV))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("null", [0, -1])
def test_varlen_ragged_partial_chunks(dtype, null):
    """Packed sequences with ragged tails, unaligned computed prefixes
    (partial first chunks), an empty sequence, mixed initial states; several
    tiles per chunk; "all" cache mode."""
    new = [300, 1, 0, 129, 64, 517]
    nc = [10, 64, 0, 63, 0, 200]
    has = [True, True, False, False, False, True]
    case = W.prefill_case(11, new, nc, 4, 64, 128, 2, 64, dtype=dtype, device=DEV, has_init=has,
                          null_block_id=null, num_slots=200)
    _run_and_check(case)


def test_default_mode_one_slot_per_sequence():
    new = [100, 260, 7]
    case = W.prefill_case(12, new, [5, 0, 33], 6, 64, 128, 3, 128, device=DEV,
                          has_init=[True, False, True], mode="default", num_slots=8)
    _run_and_check(case)


def test_small_dims_no_D_no_bias_and_dt_limit():
    case = W.prefill_case(13, [90, 45], [0, 3], 2, 16, 32, 1, 32, device=DEV, has_init=[False, True],
                          num_slots=20)
    _run_and_check(case, D=None, dt_bias=None, dt_limit=(0.05, 0.4))


@pytest.mark.parametrize("with_init", [False, True])
def test_warmup_shape_single_chunk_2048(with_init):
    """seqlen = chunk_size = 2048, H=48, P=64, N=128, G=4, bf16, with and without initial state."""
    _run_and_check(W.warmup_shape_prefill(DEV, with_init=with_init))


def test_varlen_prefix_cached_full_size_sampled_heads():
    """32 requests, U(64,4096) new tokens, U(0,8192) computed, chunk 256, half
    resuming from a [4096,48,64,128] cache; y and every chunk state checked on
    heads sampled across all groups, untouched slots checked bitwise."""
    case = W.varlen_prefix_cached_prefill(DEV)
    fp_before = PT.slot_fingerprints(case["cache"])
    before = case["cache"].clone()
    err = _err()
    y, meta = PT.run_prefill(case, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    e_y, e_s, same, tol = PT.check_prefill(case, y, meta, before, case["cache"], heads=[0, 13, 26, 47])
    assert e_y <= tol and e_s <= tol and same, (e_y, e_s, same)


def test_long_context_prefill_full_size_sampled_heads():
    """8 x 65536 fresh tokens, chunk 256, H=128, G=8, 16384-slot cache: y and
    all 2048 chunk states on two heads; fingerprints of the other slots."""
    pre, _ = W.long_mixed(DEV)
    fp_before = PT.slot_fingerprints(pre["cache"])
    err = _err()
    y, meta = PT.run_prefill(pre, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    heads = [5, 122]
    yo, cso = PT.oracle_prefill(pre, meta, pre["cache"], heads=heads)
    hs = torch.tensor(heads)
    tol = PT.TOL[torch.bfloat16]
    assert PT.y_err(y[:, hs].double().cpu().numpy(), yo, torch.bfloat16) <= tol
    sl = torch.from_numpy(meta["chunk_slot"].astype(np.int64)).to(DEV)
    assert PT.rel_err(pre["cache"][sl][:, hs].double().cpu().numpy(), cso) <= tol
    fp_after = PT.slot_fingerprints(pre["cache"])
    mask = torch.ones_like(fp_after, dtype=torch.bool)
    mask[sl] = False
    assert torch.equal(fp_after[mask], fp_before[mask])


def test_restart_from_stored_boundary_equals_one_pass():
    """Prefix caching end to end on the GPU: prefill 3 chunks, then resume the
    rest from the stored boundary state; matches one prefill over all tokens."""
    Q = 128
    full = W.prefill_case(14, [3 * Q + 77], [0], 4, 64, 128, 2, Q, device=DEV, num_slots=16)
    y_full, meta_full = PT.run_prefill(full)
    torch.cuda.synchronize()
    cache_full = full["cache"].clone()
    # same tokens, two calls
    part = dict(full)
    part["cache"] = W.sentinel_cache(16, 4, 64, 128, DEV)
    first = dict(part, x=full["x"][:3 * Q], dt=full["dt"][:3 * Q], B=full["B"][:3 * Q], C=full["C"][:3 * Q],
                 cu_seqlens=torch.tensor([0, 3 * Q], dtype=torch.int32))
    y1, m1 = PT.run_prefill(first)
    second = dict(part, x=full["x"][3 * Q:].contiguous(), dt=full["dt"][3 * Q:].contiguous(),
                  B=full["B"][3 * Q:].contiguous(), C=full["C"][3 * Q:].contiguous(),
                  cu_seqlens=torch.tensor([0, 77], dtype=torch.int32),
                  num_computed=torch.tensor([3 * Q], dtype=torch.int32), has_init=torch.tensor([True]))
    y2, m2 = PT.run_prefill(second)
    torch.cuda.synchronize()
    tol = PT.TOL[torch.bfloat16]
    assert PT.y_err(torch.cat([y1, y2]).double().cpu(), y_full.double().cpu(), torch.bfloat16) <= tol
    last = int(full["block_table"][0, 3])
    assert PT.rel_err(part["cache"][last].double().cpu(), cache_full[last].double().cpu()) <= tol


def test_out_of_range_slot_is_reported_and_skipped():
    case = W.prefill_case(15, [70], [0], 2, 16, 16, 1, 32, device=DEV, num_slots=10)
    meta = PT.prefill_metadata(case)
    meta["chunk_slot"][1] = 999
    before = case["cache"].clone()
    err = _err()
    PT.run_prefill(case, meta=meta, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ssd.DEVERR_SLOT
    keep = [s for s in range(10) if s not in (int(meta["chunk_slot"][0]), int(meta["chunk_slot"][2]))]
    assert torch.equal(case["cache"][keep].view(torch.int32), before[keep].view(torch.int32))


def test_inconsistent_metadata_is_reported():
    case = W.prefill_case(16, [40, 40], [0, 0], 2, 16, 16, 1, 32, device=DEV, num_slots=10)
    meta = PT.prefill_metadata(case)
    meta["last_chunk_indices"][0] = 0  # sequence 0 really has two chunks
    err = _err()
    PT.run_prefill(case, meta=meta, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ssd.DEVERR_METADATA


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_output_gate(dtype):
    """The output gate z: y * silu(z) on the ragged varlen batch (the
    tensor-core kernel for bf16, the CUDA-core kernels for fp32), with z wide
    enough (3 N(0,1)) to reach both tails of silu."""
    new = [300, 1, 0, 129, 64, 517]
    nc = [10, 64, 0, 63, 0, 200]
    has = [True, True, False, False, False, True]
    case = W.prefill_case(12, new, nc, 4, 64, 128, 2, 64, dtype=dtype, device=DEV, has_init=has,
                          null_block_id=0, num_slots=200)
    g = torch.Generator(device=DEV).manual_seed(99)
    z = (3.0 * torch.randn(case["x"].shape, generator=g, device=DEV)).to(dtype)
    _run_and_check(case, z=z)
