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


@pytest.mark.parametrize("Q", [96, 200, 384, 1024])
def test_tensor_core_path_chunk_sizes_off_the_block(Q):
    """Chunk sizes that are not 128: blocks never cross a chunk end, so chunks of 96 or 200 tokens
    make every block short, and 384 or 1024 put several blocks in a chunk; with unaligned computed
    prefixes (partial first chunks), initial states and ragged tails."""
    new = [700, 5, 333, 1500]
    nc = [0, 17, Q - 1, 3 * Q + 5]
    case = W.prefill_case(50 + Q, new, nc, 4, 64, 128, 2, Q, device=DEV, has_init=[False, True, True, True],
                          num_slots=80)
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


@pytest.mark.parametrize("P,N,dtype", [(128, 128, torch.bfloat16), (256, 64, torch.float32), (64, 256, torch.bfloat16)])
def test_largest_cuda_core_shapes(P, N, dtype):
    """The CUDA-core path at the largest headdim x dstate it takes (P N = 16384), varlen with
    initial states and ragged chunks."""
    case = W.prefill_case(40 + P, [300, 97], [0, 130], 2, P, N, 1, 64, dtype=dtype, device=DEV,
                          has_init=[False, True], num_slots=24)
    _run_and_check(case)


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


def test_tensor_core_path_without_D_and_bias_with_dt_limit():
    """The tensor-core kernel (bf16, headdim 64, dstate 128) with D and
    dt_bias absent and a dt_limit clamp that binds at both ends, on the ragged
    batch (partial blocks, unaligned first chunks, an empty sequence)."""
    new = [300, 1, 0, 129, 64, 517]
    nc = [10, 64, 0, 63, 0, 200]
    case = W.prefill_case(17, new, nc, 4, 64, 128, 2, 64, device=DEV,
                          has_init=[True, True, False, False, False, True], num_slots=200)
    _run_and_check(case, D=None, dt_bias=None, dt_limit=(0.05, 0.4))


def test_tensor_core_path_large_delta():
    """Step sizes of 200-300 (dt + dt_bias far above 15, the branch where
    softplus is the identity) with slow decay rates A = -exp(U(-7,-5)), so a
    token's contribution survives a few tokens: the fp16 operands P (up to
    about |C.B| * delta, ~2e4), w x and the carried state run near, but
    inside, the fp16 range."""
    case = W.prefill_case(18, [700, 190], [0, 0], 4, 64, 128, 2, 256, device=DEV, num_slots=40)
    g = torch.Generator(device=DEV).manual_seed(5)
    case["A"] = -torch.exp(-7.0 + 2.0 * torch.rand(4, generator=g, device=DEV))
    bias = 200.0 + 100.0 * torch.rand(4, generator=g, device=DEV)
    _run_and_check(case, dt_bias=bias)


def test_tensor_core_path_decay_beyond_the_factored_range():
    """Per-token decays delta |A| of about 40, 6, 1 and 0.1 for the four heads (dt_bias 2): a
    32-token group then decays by about 1300, 200, 34 and 3 in the log domain.  The first two heads
    exceed the range where the P pass factors exp(c_t - c_s) into a row and a column factor (80),
    so their diagonal groups take one exponential per element; the others take the factored form."""
    case = W.prefill_case(20, [700, 190], [0, 0], 4, 64, 128, 2, 256, device=DEV, num_slots=40)
    case["A"] = torch.tensor([-20.0, -3.0, -0.5, -0.05], device=DEV)
    bias = torch.full((4,), 2.0, device=DEV)
    _run_and_check(case, dt_bias=bias)


def test_non_finite_tokens_of_the_next_sequence_stay_out():
    """The last block of sequence 0 is short (200 = 128 + 72 tokens), so the
    128-row tiles of that block also hold sequence 1's first 56 tokens.  Those
    hold inf and NaN in x, B, C and dt: sequence 0's y and stored states must
    stay finite and at parity with the oracle on sequence 0 alone."""
    case = W.prefill_case(19, [200, 300], [0, 0], 4, 64, 128, 2, 256, device=DEV, num_slots=40)
    ref = {k: case[k].clone() for k in ("x", "B", "C", "dt")}
    case["x"][200:256] = float("nan")
    case["x"][230:240, 1] = float("inf")
    case["B"][200:256] = float("inf")
    case["B"][220:230, 0] = -float("inf")
    case["C"][200:256] = float("nan")
    case["dt"][200:256] = float("inf")
    before = case["cache"].clone()
    err = _err()
    y, meta = PT.run_prefill(case, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    k0 = int(meta["last_chunk_indices"][0]) + 1  # chunks of sequence 0
    assert torch.isfinite(y[:200]).all()
    slots0 = [int(s) for s in meta["chunk_slot"][:k0]]
    assert torch.isfinite(case["cache"][slots0]).all()
    # oracle on sequence 0 alone, with its (finite) tokens
    one = dict(case, x=ref["x"][:200], B=ref["B"][:200], C=ref["C"][:200], dt=ref["dt"][:200],
               cu_seqlens=torch.tensor([0, 200], dtype=torch.int32))
    m0 = {"cu_chunk_seqlens": meta["cu_chunk_seqlens"][:k0 + 1], "init_slot": meta["init_slot"][:1]}
    yo, cso = PT.oracle_prefill(one, m0, before)
    tol = PT.TOL[torch.bfloat16]
    assert PT.y_err(y[:200].double().cpu().numpy(), yo, torch.bfloat16) <= tol
    assert PT.rel_err(case["cache"][slots0].double().cpu().numpy(), cso) <= tol


def test_repeated_seq_order_entry_is_reported():
    case = W.prefill_case(20, [150, 90], [0, 0], 4, 64, 128, 2, 64, device=DEV, num_slots=20)
    meta = PT.prefill_metadata(case)
    meta["seq_order"] = np.array([0, 0], np.int32)
    err = _err()
    PT.run_prefill(case, meta=meta, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ssd.DEVERR_METADATA


def test_bounded_waits_give_up_and_the_context_survives():
    """With a watchdog of 100 cycles every CTA's first wait for a tile gives
    up: the call returns, SSD_DEVERR_TIMEOUT is set, and the next call (the
    default watchdog) on the same context is correct."""
    case = W.prefill_case(21, [300, 129], [0, 0], 4, 64, 128, 2, 64, device=DEV, num_slots=40)
    err = _err()
    PT.run_prefill(case, err=err, wait_limit_cycles=100)
    torch.cuda.synchronize()
    assert int(err.item()) & ssd.DEVERR_TIMEOUT
    case["cache"] = W.sentinel_cache(40, 4, 64, 128, DEV)
    _run_and_check(case)


@pytest.mark.parametrize("gate", [False, True])
def test_sequences_split_across_ctas(gate):
    """Two sequences and eight heads are too few (sequence, head) pairs to fill the GPU, so each
    sequence is cut into segments of whole blocks that separate CTAs run: the long sequence's
    segments start mid-chunk from the state the segment pass carries in; the short one (one
    block) leaves most of its segments empty.  Initial states, unaligned computed prefixes,
    "all" mode, with and without the output gate; y and every stored state against the oracle."""
    case = W.prefill_case(22, [2000, 100], [37, 300], 8, 64, 128, 2, 256, device=DEV,
                          has_init=[True, True], num_slots=64)
    t = {k: torch.from_numpy(v).to(DEV) for k, v in PT.prefill_metadata(case).items()}
    a = ssd.prefill_args(case["x"], case["dt"], case["A"], case["B"], case["C"], case["cu_seqlens"].to(DEV),
                         t["cu_chunk_seqlens"], t["seq_idx"], t["last_chunk_indices"], torch.empty_like(case["x"]))
    assert ssd.ssd_prefill_kernel_count(a) == 3  # the segment pass runs
    if gate:
        g = torch.Generator(device=DEV).manual_seed(7)
        _run_and_check(case, z=(3.0 * torch.randn(case["x"].shape, generator=g, device=DEV)).to(case["x"].dtype))
    else:
        _run_and_check(case)


def test_one_sequence_split_into_eight_segments():
    """One 8192-token sequence and four heads: the split reaches its maximum of eight segments
    (SMs / heads and tokens / 256 both allow more), so segment 7 starts from segment 0's end state
    carried through six segment decays.  An initial state, "all" mode, chunk 256; y and all 32
    chunk states against the oracle."""
    case = W.prefill_case(23, [8192], [512], 4, 64, 128, 2, 256, device=DEV, has_init=[True], num_slots=48)
    t = {k: torch.from_numpy(v).to(DEV) for k, v in PT.prefill_metadata(case).items()}
    a = ssd.prefill_args(case["x"], case["dt"], case["A"], case["B"], case["C"], case["cu_seqlens"].to(DEV),
                         t["cu_chunk_seqlens"], t["seq_idx"], t["last_chunk_indices"], torch.empty_like(case["x"]))
    assert ssd.ssd_prefill_kernel_count(a) == 3
    _run_and_check(case)


@pytest.mark.parametrize("P", [64, 32])
def test_marked_call_records_its_event_and_changes_nothing(P):
    """ssd_prefill_varlen_marked records the caller's event before the main kernel (after the prep
    kernel on the tensor-core path, before everything on the CUDA-core path) and gives the bits of
    the plain call."""
    case = W.prefill_case(60 + P, [700, 300], [0, 40], 4, P, 128, 2, 256, device=DEV, has_init=[False, True],
                          num_slots=24)
    before = case["cache"].clone()
    y0, meta = PT.run_prefill(case)
    torch.cuda.synchronize()
    after = case["cache"].clone()
    case["cache"].copy_(before)
    start, mark, end = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    start.record()
    y1, _ = PT.run_prefill(case, meta=meta, mark=mark)
    end.record()
    torch.cuda.synchronize()
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    assert torch.equal(after.view(torch.int32), case["cache"].view(torch.int32))
    assert start.elapsed_time(mark) >= 0 and mark.elapsed_time(end) > 0
