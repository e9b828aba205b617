"""Host-side checks of the C ABI that need no GPU: the library loads and
exports every symbol the header declares, the host chunk metadata matches the
oracle's per-token definition bit for bit, and invalid arguments are refused
before anything is launched."""
import ctypes
import os
import re

import numpy as np
import pytest

import selective_state_space_mamba2_gb300 as ssd
from selective_state_space_mamba2_gb300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    ssd.build()
    return ssd.lib()


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"SSD_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)
    return names


def test_library_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert set(B.EXPORTED_SYMBOLS) <= set(declared)
    for name in declared:
        assert hasattr(lib, name), name
    assert lib.ssd_abi_version() == 2
    assert lib.ssd_status_string(3) == b"SSD_ERR_WORKSPACE"


def test_max_chunks_bound(lib):
    assert ssd.ssd_max_chunks(1, 0, 4) == 0
    assert ssd.ssd_max_chunks(2, 4, 4) == 4
    assert ssd.ssd_max_chunks(3, 100, 16) == 6 + 7
    assert ssd.ssd_max_chunks(-1, 5, 4) == -1


@pytest.mark.parametrize("seed", range(30))
def test_metadata_matches_oracle_bit_exact(lib, oracle_lib, seed):
    rng = np.random.default_rng(seed)
    S = int(rng.integers(1, 40))
    Q = int(rng.choice([1, 5, 16, 64, 256, 2048]))
    lens = rng.integers(0, 4 * Q + 9, S)
    nc = rng.integers(0, 8 * Q + 3, S)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    has = rng.integers(0, 2, S).astype(bool) & (nc > 0)
    null = int(rng.choice([0, -1]))
    cols = int(((nc + lens - 1) // Q).max()) + 2
    bt = rng.permutation(np.arange(1, S * cols + 1)).reshape(S, cols).astype(np.int32)
    m = ssd.ssd_chunk_metadata(cu, Q, nc, has, block_table=bt, null_block_id=null)
    o = oracle_lib.chunk_metadata(cu, nc, Q)
    for key in ("cu_chunk_seqlens", "seq_idx", "last_chunk_indices", "chunk_block_col"):
        assert np.array_equal(m[key], o[key]), key
    init, cslot = oracle_lib.prefill_slots(o, nc, Q, null, block_table=bt, has_initial_states=has)
    assert np.array_equal(m["init_slot"], init) and np.array_equal(m["chunk_slot"], cslot)
    si = rng.permutation(np.arange(1, S + 1)).astype(np.int32)
    md = ssd.ssd_chunk_metadata(cu, Q, nc, has, state_indices=si, null_block_id=null)
    init_d, cslot_d = oracle_lib.prefill_slots(o, nc, Q, null, state_indices=si, has_initial_states=has)
    assert np.array_equal(md["init_slot"], init_d) and np.array_equal(md["chunk_slot"], cslot_d)


def test_seq_order_is_longest_first_permutation(lib):
    cu = np.array([0, 5, 5, 30, 31, 40, 65], np.int32)  # lengths 5, 0, 25, 1, 9, 25
    m = ssd.ssd_chunk_metadata(cu, 8)
    assert m["seq_order"].tolist() == [2, 5, 4, 0, 3, 1]


def test_metadata_rejects_bad_input(lib):
    with pytest.raises(B.SSDError) as e:
        ssd.ssd_chunk_metadata([0, 5, 3], 4)
    assert e.value.code == B.SSD_ERR_INVALID_ARG
    with pytest.raises(B.SSDError):
        ssd.ssd_chunk_metadata([1, 5], 4)
    with pytest.raises(B.SSDError):
        ssd.ssd_chunk_metadata([0, 5], 0)
    with pytest.raises(B.SSDError):  # initial state but nothing computed ("all" mode)
        ssd.ssd_chunk_metadata([0, 5], 4, [0], [True], block_table=np.ones((1, 4), np.int32))
    with pytest.raises(B.SSDError):  # block column beyond the table
        ssd.ssd_chunk_metadata([0, 9], 4, [0], block_table=np.ones((1, 2), np.int32))


def _prefill_args(**over):
    a = B.PrefillArgs()
    a.total_tokens, a.num_seqs, a.num_chunks = 8, 1, 1
    a.nheads, a.headdim, a.dstate, a.ngroups, a.chunk_size = 2, 4, 4, 1, 8
    a.dtype, a.dt_softplus, a.dt_min, a.dt_max = B.SSD_F32, 1, 0.0, float("inf")
    for f in ("x", "dt", "B", "C", "A", "y", "cu_seqlens", "cu_chunk_seqlens", "last_chunk_indices"):
        setattr(a, f, 0x10000)
    for k, v in over.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("over,code", [
    (dict(ngroups=3), B.SSD_ERR_INVALID_ARG),
    (dict(headdim=257), B.SSD_ERR_INVALID_ARG),
    (dict(dtype=7), B.SSD_ERR_INVALID_ARG),
    (dict(z=0x20008), B.SSD_ERR_INVALID_ARG),  # the gate must be 16-byte aligned too
    (dict(x=0x10008), B.SSD_ERR_INVALID_ARG),
    (dict(x=None), B.SSD_ERR_INVALID_ARG),
    (dict(dt_min=1.0, dt_max=0.5), B.SSD_ERR_INVALID_ARG),
    (dict(num_chunks=0), B.SSD_ERR_INVALID_ARG),
    (dict(init_slot=0x10000), B.SSD_ERR_INVALID_ARG),  # slots without a cache
    (dict(wait_limit_cycles=-1), B.SSD_ERR_INVALID_ARG),
])
def test_prefill_host_validation(lib, over, code):
    a = _prefill_args(**over)
    assert lib.ssd_prefill_varlen(ctypes.byref(a), None, 0, None) == code
    assert lib.ssd_prefill_varlen_marked(ctypes.byref(a), None, 0, None, None) == code
    assert lib.ssd_prefill_workspace_size(ctypes.byref(a)) == 0


def test_prefill_beyond_the_cuda_core_path_is_unsupported(lib):
    # headdim x dstate above 16384 (the CUDA-core kernels' per-CTA state), not a tensor-core shape
    a = _prefill_args(headdim=256, dstate=256)
    assert lib.ssd_prefill_varlen(ctypes.byref(a), ctypes.c_void_p(0x100000), 1 << 40, None) == B.SSD_ERR_UNSUPPORTED


def test_prefill_workspace_too_small_is_refused(lib):
    a = _prefill_args()
    need = lib.ssd_prefill_workspace_size(ctypes.byref(a))
    assert need > 0
    assert lib.ssd_prefill_varlen(ctypes.byref(a), ctypes.c_void_p(0x100000), need - 1, None) == B.SSD_ERR_WORKSPACE
    assert lib.ssd_prefill_varlen(ctypes.byref(a), ctypes.c_void_p(0x100010), need, None) == B.SSD_ERR_WORKSPACE


def _up256(n):
    return (n + 255) // 256 * 256


@pytest.mark.parametrize("T,H,K,P,N", [(8, 2, 1, 4, 4), (2048, 48, 1, 64, 128), (3, 1, 3, 8, 16), (1000, 48, 5, 64, 128)])
def test_cuda_core_workspace_is_the_documented_formula(lib, T, H, K, P, N):
    """ssd.h gives the CUDA-core path's scratch as up256(4HT) + up256(8HT) + 2 up256(4KHPN);
    one 2048-token chunk at H=48, P=64, N=128 is its "about 4.3 MB" example."""
    a = _prefill_args(total_tokens=T, nheads=H, num_chunks=K, headdim=P, dstate=N)
    need = lib.ssd_prefill_workspace_size(ctypes.byref(a))
    assert need == _up256(4 * H * T) + _up256(8 * H * T) + 2 * _up256(4 * K * H * P * N)
    if (T, H, K) == (2048, 48, 1):
        assert round(need / 1e6, 1) == 4.3


@pytest.mark.parametrize("T,G", [(1, 1), (777, 8), (65536, 8)])
def test_tensor_core_workspace_is_the_documented_formula(lib, T, G):
    """bf16 with headdim 64 and dstate 128: fp16 copies of B and C plus delta and its in-block
    cumsum per head and token, 2 up256(2 T G N) + 2 up256(4 H T) bytes."""
    a = _prefill_args(total_tokens=T, nheads=2 * G, ngroups=G, headdim=64, dstate=128, dtype=B.SSD_BF16)
    assert lib.ssd_prefill_kernel_count(ctypes.byref(a)) == 2
    assert lib.ssd_prefill_workspace_size(ctypes.byref(a)) == 2 * _up256(2 * T * G * 128) + 2 * _up256(4 * 2 * G * T)


def test_noalloc_refusal_is_decided_on_the_host(lib):
    # 40 chunks of states at H=48, P=64, N=128 need 2 * 40 * 1.57 MB of scratch, beyond 64 MiB
    a = _prefill_args(total_tokens=2048, num_chunks=40, nheads=48, headdim=64, dstate=128)
    assert lib.ssd_prefill_workspace_size(ctypes.byref(a)) > 64 << 20
    assert lib.ssd_prefill_varlen_noalloc(ctypes.byref(a), None) == B.SSD_ERR_WORKSPACE


def test_empty_prefill_is_a_no_op(lib):
    a = _prefill_args(total_tokens=0, num_chunks=0)
    assert lib.ssd_prefill_varlen(ctypes.byref(a), None, 0, None) == B.SSD_OK


def _decode_args(**over):
    a = B.DecodeArgs()
    a.batch, a.tokens_per_req, a.nheads, a.headdim, a.dstate, a.ngroups = 2, 1, 2, 4, 8, 1
    a.dtype, a.dt_softplus, a.dt_min, a.dt_max = B.SSD_BF16, 1, 0.0, float("inf")
    a.num_slots, a.null_block_id, a.state_indices_cols = 4, 0, 1
    for f in ("x", "dt", "B", "C", "A", "y", "state_cache", "state_indices"):
        setattr(a, f, 0x10000)
    for k, v in over.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("over,code", [
    (dict(tokens_per_req=0), B.SSD_ERR_INVALID_ARG),
    (dict(tokens_per_req=2), B.SSD_ERR_INVALID_ARG),  # fewer columns than tokens
    (dict(ngroups=3), B.SSD_ERR_INVALID_ARG),
    (dict(state_cache=0x10004), B.SSD_ERR_INVALID_ARG),
    (dict(dstate=6), B.SSD_ERR_INVALID_ARG),
    (dict(dstate=12), B.SSD_ERR_UNSUPPORTED),
    (dict(num_slots=0), B.SSD_ERR_INVALID_ARG),
])
def test_decode_host_validation(lib, over, code):
    a = _decode_args(**over)
    assert lib.ssm_decode_update(ctypes.byref(a), None) == code


def test_empty_decode_is_a_no_op(lib):
    a = _decode_args(batch=0)
    assert lib.ssm_decode_update(ctypes.byref(a), None) == B.SSD_OK


@pytest.mark.parametrize("pre,dec,code", [
    (dict(ngroups=3), {}, B.SSD_ERR_INVALID_ARG),       # a bad prefill part
    ({}, dict(tokens_per_req=0), B.SSD_ERR_INVALID_ARG),  # a bad decode part
    ({}, dict(dstate=12), B.SSD_ERR_UNSUPPORTED),
    (dict(headdim=257), dict(batch=0), B.SSD_ERR_INVALID_ARG),  # checked even beside an empty part
    (dict(total_tokens=0, num_chunks=0), dict(state_cache=0x10004), B.SSD_ERR_INVALID_ARG),
])
def test_mixed_step_checks_both_parts_before_queueing(lib, pre, dec, code):
    """ssd_mixed_step makes the host checks of both calls before anything is queued, so a bad
    part is refused on a machine without a GPU."""
    a, d = _prefill_args(**pre), _decode_args(**dec)
    assert lib.ssd_mixed_step(ctypes.byref(a), None, 0, ctypes.byref(d), None) == code


def test_mixed_step_refuses_a_short_workspace_before_queueing(lib):
    a, d = _prefill_args(), _decode_args()
    need = lib.ssd_prefill_workspace_size(ctypes.byref(a))
    assert lib.ssd_mixed_step(ctypes.byref(a), ctypes.c_void_p(0x100000), need - 1, ctypes.byref(d), None) \
        == B.SSD_ERR_WORKSPACE


def test_empty_mixed_step_is_a_no_op(lib):
    a, d = _prefill_args(total_tokens=0, num_chunks=0), _decode_args(batch=0)
    assert lib.ssd_mixed_step(ctypes.byref(a), None, 0, ctypes.byref(d), None) == B.SSD_OK


def _conv_args(**over):
    a = B.Conv1dArgs()
    a.total_tokens, a.num_seqs, a.num_chunks, a.tokens_per_req = 8, 2, 0, 4
    a.dim_x, a.dim_bc, a.width, a.dtype, a.activation = 16, 8, 4, B.SSD_BF16, 1
    a.num_slots, a.null_block_id = 4, 0
    for f in ("xbc", "weight", "cu_seqlens", "x_out", "B_out", "C_out", "conv_state", "init_slot"):
        setattr(a, f, 0x10000)
    for k, v in over.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("over,code", [
    (dict(dim_x=12), B.SSD_ERR_INVALID_ARG),       # channels in groups of 8 (16-byte vectors)
    (dict(width=5), B.SSD_ERR_INVALID_ARG),
    (dict(width=1), B.SSD_ERR_INVALID_ARG),
    (dict(activation=2), B.SSD_ERR_INVALID_ARG),
    (dict(dtype=7), B.SSD_ERR_INVALID_ARG),
    (dict(xbc=0x10008), B.SSD_ERR_INVALID_ARG),
    (dict(weight=0x10004), B.SSD_ERR_INVALID_ARG),  # weight rows are read in 16-byte pieces
    (dict(cu_seqlens=None), B.SSD_ERR_INVALID_ARG),
    (dict(conv_state=None), B.SSD_ERR_INVALID_ARG),  # slots without a state tensor
    (dict(chunk_slot=0x10000), B.SSD_ERR_INVALID_ARG),  # chunk slots without chunk metadata
])
def test_conv1d_host_validation(lib, over, code):
    a = _conv_args(**over)
    assert lib.ssd_conv1d_varlen(ctypes.byref(a), None) == code


@pytest.mark.parametrize("over,code", [
    (dict(tokens_per_req=3), B.SSD_ERR_INVALID_ARG),  # 2 requests x 3 tokens != 8 rows
    (dict(tokens_per_req=0), B.SSD_ERR_INVALID_ARG),
    (dict(init_slot=None), B.SSD_ERR_INVALID_ARG),   # decode needs the request slots
])
def test_conv1d_update_host_validation(lib, over, code):
    a = _conv_args(**over)
    assert lib.ssd_conv1d_update(ctypes.byref(a), None) == code


def test_empty_conv1d_is_a_no_op(lib):
    a = _conv_args(total_tokens=0, num_seqs=0)
    assert lib.ssd_conv1d_varlen(ctypes.byref(a), None) == B.SSD_OK
    assert lib.ssd_conv1d_update(ctypes.byref(a), None) == B.SSD_OK


def _m1_args(**over):
    a = B.Mamba1Args()
    a.total_tokens, a.num_seqs, a.num_chunks, a.tokens_per_req = 8, 2, 2, 4
    a.dim, a.dstate, a.ngroups, a.dtype, a.dt_softplus = 128, 16, 1, B.SSD_BF16, 1
    a.dt_min, a.dt_max = 0.0, float("inf")
    a.num_slots, a.null_block_id, a.state_indices_cols = 4, 0, 4
    for f in ("x", "dt", "B", "C", "A", "y", "cu_seqlens", "cu_chunk_seqlens", "last_chunk_indices",
              "state_cache", "state_indices", "init_slot"):
        setattr(a, f, 0x10000)
    for k, v in over.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("over,code", [
    (dict(dim=96), B.SSD_ERR_UNSUPPORTED),          # channels in CTAs of 64
    (dict(dstate=4), B.SSD_ERR_UNSUPPORTED),        # dstate 8 or 16
    (dict(ngroups=4), B.SSD_ERR_UNSUPPORTED),       # 32 channels per group: a CTA would span groups
    (dict(ngroups=3), B.SSD_ERR_INVALID_ARG),       # groups must divide the channels
    (dict(dtype=7), B.SSD_ERR_INVALID_ARG),
    (dict(dt_min=2.0, dt_max=1.0), B.SSD_ERR_INVALID_ARG),
    (dict(x=0x10008), B.SSD_ERR_INVALID_ARG),       # 16-byte copies of x rows
    (dict(dt=0x10004), B.SSD_ERR_INVALID_ARG),
    (dict(cu_chunk_seqlens=None), B.SSD_ERR_INVALID_ARG),
    (dict(num_chunks=0), B.SSD_ERR_INVALID_ARG),    # tokens without chunks
    (dict(state_cache=None), B.SSD_ERR_INVALID_ARG),  # initial-state slots without a cache
])
def test_mamba1_scan_host_validation(lib, over, code):
    a = _m1_args(**over)
    assert lib.mamba1_scan_varlen(ctypes.byref(a), None) == code


@pytest.mark.parametrize("over,code", [
    (dict(tokens_per_req=3), B.SSD_ERR_INVALID_ARG),     # 2 requests x 3 tokens != 8 rows
    (dict(state_indices_cols=3), B.SSD_ERR_INVALID_ARG),  # fewer columns than tokens per request
    (dict(state_indices=None), B.SSD_ERR_INVALID_ARG),
    (dict(state_cache=None), B.SSD_ERR_INVALID_ARG),
    (dict(dstate=32), B.SSD_ERR_UNSUPPORTED),
    (dict(A=0x10004), B.SSD_ERR_INVALID_ARG),  # A rows are read in 16-byte pieces
])
def test_mamba1_update_host_validation(lib, over, code):
    a = _m1_args(**over)
    assert lib.mamba1_state_update(ctypes.byref(a), None) == code


def test_empty_mamba1_is_a_no_op(lib):
    a = _m1_args(total_tokens=0, num_seqs=0, num_chunks=0)
    assert lib.mamba1_scan_varlen(ctypes.byref(a), None) == B.SSD_OK
    assert lib.mamba1_state_update(ctypes.byref(a), None) == B.SSD_OK


def test_calls_fail_loudly_without_the_library(monkeypatch, tmp_path):
    """There is no implementation behind the binding but the CUDA library: without it every call
    raises instead of computing anything."""
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(B, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        ssd.ssd_max_chunks(1, 8, 4)
    with pytest.raises(RuntimeError, match="missing"):
        ssd.ssd_chunk_metadata([0, 5], 4)
    with pytest.raises(RuntimeError, match="missing"):
        B.lib()


def test_device_calls_refuse_host_tensors():
    """Host (CPU) tensors are refused by every device call: there is no CPU path to fall back to."""
    import torch
    R, H, P, N = 2, 2, 4, 8
    x = torch.zeros(R, H, P, dtype=torch.bfloat16)
    dt = torch.zeros(R, H, dtype=torch.bfloat16)
    Bm = torch.zeros(R, 1, N, dtype=torch.bfloat16)
    A = torch.full((H,), -1.0)
    cache = torch.zeros(4, H, P, N)
    si = torch.ones(R, 1, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ssd.ssm_decode_update(x, dt, A, Bm, Bm, cache, si)
    cu = torch.tensor([0, R], dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ssd.ssd_prefill_varlen(x, dt, A, Bm, Bm, cu, cu, torch.zeros(1, dtype=torch.int32),
                               torch.zeros(1, dtype=torch.int32))
