"""Seeded synthetic inputs for the SSD prefill and SSM decode calls.

This module only draws numbers: token tensors, per-head parameters, sequence
lengths, computed-token counts, initial-state flags, slot tables and cache
contents.  It holds none of the recurrence's arithmetic, so both the CUDA
path and the CPU oracle may consume what it produces.

The shapes follow the varlen chunk-scan call shown on "[vllm] vLLM Mamba2 SSD
커널 웜업" (section "mamba_mixer2.py 변경 사항 (핵심)"): x [T,H,P], dt [T,H],
B and C [T,G,N], per-head A, D and dt_bias, and an fp32 state cache
[slots, H, P, N] whose shape per slot matches the SSM state of
"vLLM v0.20.0 하이브리드 SSM 모델을 위한 분산 서빙 추가" (section "전체 흐름:
Nemotron-H 예시": [num_blocks, 48, 64, 128]).

Distributions: x, B, C, dt ~ N(0,1) (randn, as the warm-up call uses, not
zeros); A = -exp(U(0,2)); D ~ N(0,1); dt_bias ~ U(-4,-1) unless a case fixes
it; cache slots that are read hold N(0,1); every other slot holds the
SENTINEL bit pattern so that a stray write is visible bit for bit.
"""
from __future__ import annotations

import torch

# quiet NaN with a payload: visible in bitwise compares, poisons any read
SENTINEL_BITS = 0x7FC0DEAD


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def sentinel_cache(num_slots, H, P, N, device):
    return torch.full((num_slots, H, P, N), SENTINEL_BITS, dtype=torch.int32,
                      device=device).view(torch.float32)


def head_params(H, device, seed, dt_bias_range=(-4.0, -1.0), dt_bias_zero=False):
    g = _gen(device, seed + 7919)
    A = -torch.exp(torch.rand(H, generator=g, device=device) * 2.0)
    D = torch.randn(H, generator=g, device=device)
    if dt_bias_zero:
        dt_bias = torch.zeros(H, device=device)
    else:
        lo, hi = dt_bias_range
        dt_bias = lo + (hi - lo) * torch.rand(H, generator=g, device=device)
    return A.float(), D.float(), dt_bias.float()


def tokens(T, H, P, N, G, dtype, device, seed):
    g = _gen(device, seed)
    x = torch.randn(T, H, P, generator=g, device=device).to(dtype)
    dt = torch.randn(T, H, generator=g, device=device).to(dtype)
    B = torch.randn(T, G, N, generator=g, device=device).to(dtype)
    C = torch.randn(T, G, N, generator=g, device=device).to(dtype)
    return x, dt, B, C


def prefill_case(seed, new_tokens, num_computed, H, P, N, G, chunk_size, dtype=torch.bfloat16,
                 device="cpu", has_init=None, num_slots=None, null_block_id=0, mode="all",
                 dt_bias_zero=False):
    """A varlen prefill batch.

    ``new_tokens`` and ``num_computed`` are per-sequence lists.  mode "all"
    draws a block table [S, cols] of distinct slots (one per chunk_size
    block, as in the "all" cache mode); mode "default" draws one distinct
    slot per sequence.  Slots are drawn from [1, num_slots) without
    replacement, so slot 0 stays free and may serve as the null id.  The
    cache holds N(0,1) in every slot some sequence reads as its initial
    state and the sentinel elsewhere.
    """
    S = len(new_tokens)
    gcpu = _gen("cpu", seed + 104729)
    cu = [0]
    for n in new_tokens:
        cu.append(cu[-1] + int(n))
    T = cu[-1]
    cu_seqlens = torch.tensor(cu, dtype=torch.int32)
    nc = torch.tensor([int(v) for v in num_computed], dtype=torch.int32)
    if has_init is None:
        has_init = [False] * S
    has = torch.tensor([bool(v) for v in has_init], dtype=torch.bool)
    cols = [((int(nc[r]) + int(new_tokens[r]) - 1) // chunk_size) + 1 if new_tokens[r] or nc[r]
            else 1 for r in range(S)]
    max_cols = max(cols) if S else 1
    if mode == "all":
        need = S * max_cols
    else:
        need = S
    if num_slots is None:
        num_slots = need + 1
    assert num_slots - 1 >= need, "not enough slots for distinct draws"
    perm = torch.randperm(num_slots - 1, generator=gcpu)[:need] + 1
    if mode == "all":
        block_table = perm.view(S, max_cols).to(torch.int32).contiguous()
        state_indices = None
    else:
        block_table = None
        state_indices = perm.to(torch.int32).contiguous()
    x, dt, B, C = tokens(T, H, P, N, G, dtype, device, seed)
    A, D, dt_bias = head_params(H, device, seed, dt_bias_zero=dt_bias_zero)
    cache = sentinel_cache(num_slots, H, P, N, device)
    gi = _gen(device, seed + 15485863)
    for r in range(S):
        if not has[r]:
            continue
        if mode == "all":
            slot = int(block_table[r, (int(nc[r]) - 1) // chunk_size])
        else:
            slot = int(state_indices[r])
        cache[slot] = torch.randn(H, P, N, generator=gi, device=device)
    return dict(x=x, dt=dt, B=B, C=C, A=A, D=D, dt_bias=dt_bias, cu_seqlens=cu_seqlens,
                num_computed=nc, has_init=has, block_table=block_table,
                state_indices=state_indices, cache=cache, chunk_size=int(chunk_size),
                null_block_id=int(null_block_id), num_slots=int(num_slots))


def decode_case(seed, live, padded, tokens_per_req, H, P, N, G, num_slots, dtype=torch.bfloat16,
                device="cpu", null_block_id=0, ncols=None, spec_accept=True):
    """A padded decode batch: ``live`` requests padded to ``padded`` rows.

    Live rows get ``ncols`` (>= tokens_per_req) distinct slots; padded rows
    are filled with null_block_id.  num_accepted_tokens ~ U{0..tokens_per_req-1}
    when ``spec_accept`` else all zero.  The slot each live request reads
    holds N(0,1); the rest of the cache holds the sentinel.
    """
    ncols = ncols or tokens_per_req
    gcpu = _gen("cpu", seed + 104729)
    need = live * ncols
    assert num_slots - 1 >= need
    perm = torch.randperm(num_slots - 1, generator=gcpu)[:need] + 1
    si = torch.full((padded, ncols), int(null_block_id), dtype=torch.int32)
    si[:live] = perm.view(live, ncols).to(torch.int32)
    if spec_accept and tokens_per_req > 1:
        na = torch.randint(0, tokens_per_req, (padded,), generator=gcpu, dtype=torch.int32)
    else:
        na = torch.zeros(padded, dtype=torch.int32)
    T = padded * tokens_per_req
    x, dt, B, C = tokens(T, H, P, N, G, dtype, device, seed)
    A, D, dt_bias = head_params(H, device, seed)
    cache = sentinel_cache(num_slots, H, P, N, device)
    gi = _gen(device, seed + 15485863)
    for r in range(live):
        cache[int(si[r, int(na[r])])] = torch.randn(H, P, N, generator=gi, device=device)
    return dict(x=x, dt=dt, B=B, C=C, A=A, D=D, dt_bias=dt_bias, state_indices=si,
                num_accepted=na, cache=cache, tokens_per_req=int(tokens_per_req),
                null_block_id=int(null_block_id), num_slots=int(num_slots), live=int(live))


# The five benchmark shapes, by what they are.

def tiny_fp32_prefill(device="cpu"):
    """1 sequence of 256 tokens, H=4, P=16, N=16, G=1, chunk 64, fp32, dt_bias=0, zero init, seed 0."""
    return prefill_case(0, [256], [0], 4, 16, 16, 1, 64, dtype=torch.float32, device=device,
                        dt_bias_zero=True, mode="default")


def warmup_shape_prefill(device="cpu", with_init=False):
    """seqlen = chunk_size = 2048, batch 1, H=48, P=64, N=128, G=4, bf16, seed 1."""
    return prefill_case(1, [2048], [2048 if with_init else 0], 48, 64, 128, 4, 2048,
                        device=device, has_init=[with_init], mode="default", num_slots=4)


def varlen_prefix_cached_prefill(device="cpu", seed=2, num_seqs=32, max_new=4096, min_new=64,
                                 max_computed=8192, num_slots=4096, H=48, P=64, N=128, G=4,
                                 chunk_size=256):
    """32 requests, new ~ U(64,4096), computed ~ U(0,8192), half with initial states, "all" mode."""
    g = _gen("cpu", seed)
    new = torch.randint(min_new, max_new + 1, (num_seqs,), generator=g).tolist()
    nc = torch.randint(0, max_computed + 1, (num_seqs,), generator=g).tolist()
    pick = torch.randperm(num_seqs, generator=g)[: num_seqs // 2].tolist()
    has = [False] * num_seqs
    for r in pick:
        if nc[r] == 0:
            nc[r] = 1 + int(torch.randint(0, max_computed, (1,), generator=g))
        has[r] = True
    return prefill_case(seed, new, nc, H, P, N, G, chunk_size, device=device, has_init=has,
                        num_slots=num_slots, mode="all")


def spec_decode_batch(device="cpu", seed=3, live=256, padded=512, tokens_per_req=4,
                      num_slots=8192, H=48, P=64, N=128, G=4):
    """256 live requests padded to 512, 1+3 tokens, num_accepted ~ U{0..3}."""
    return decode_case(seed, live, padded, tokens_per_req, H, P, N, G, num_slots, device=device)


def long_mixed(device="cpu", seed=4, num_prefills=8, prefill_len=65536, num_decodes=384,
               chunk_size=256, H=128, P=64, N=128, G=8, num_slots=16384):
    """8 fresh prefills of 65536 tokens plus 384 single-token decodes, slots distinct across both."""
    S = num_prefills
    pre = prefill_case(seed, [prefill_len] * S, [0] * S, H, P, N, G, chunk_size, device=device,
                       num_slots=num_slots, mode="all")
    used = set(int(v) for v in pre["block_table"].flatten().tolist())
    gcpu = _gen("cpu", seed + 31)
    free = [s for s in torch.randperm(num_slots - 1, generator=gcpu).add(1).tolist()
            if s not in used]
    assert len(free) >= num_decodes
    si = torch.tensor(free[:max(num_decodes, 1)], dtype=torch.int32).view(max(num_decodes, 1), 1)
    x, dt, B, C = tokens(max(num_decodes, 1), H, P, N, G, torch.bfloat16, device, seed + 1)
    gi = _gen(device, seed + 32452843)
    cache = pre["cache"]
    for r in range(num_decodes):
        cache[int(si[r, 0])] = torch.randn(H, P, N, generator=gi, device=device)
    dec = dict(x=x, dt=dt, B=B, C=C, A=pre["A"], D=pre["D"], dt_bias=pre["dt_bias"],
               state_indices=si, num_accepted=None, cache=cache, tokens_per_req=1,
               null_block_id=pre["null_block_id"], num_slots=num_slots, live=num_decodes)
    return pre, dec


# Mamba1 (per-channel states): the same draws with one channel per "head" of
# width 1, an A of shape [channels, dstate] and an optional gate z [T, channels].
# A = -exp(U(0, ln 16)): per (channel, state index) rates spread over the range
# of the S4D-real start values 1..16 that Mamba1 layers begin from.

def mamba1_A(Dc, N, device, seed):
    g = _gen(device, seed + 2750159)
    return (-torch.exp(torch.rand(Dc, N, generator=g, device=device) * 2.772588722239781)).float()


def _as_mamba1(c, N, seed, device, gate):
    T, Dc = c["x"].shape[0], c["x"].shape[1]
    c["x"] = c["x"].reshape(T, Dc)
    c["cache"] = c["cache"].reshape(c["cache"].shape[0], Dc, N)
    c["A"] = mamba1_A(Dc, N, device, seed)
    if gate:
        c["z"] = torch.randn(T, Dc, generator=_gen(device, seed + 3), device=device).to(c["x"].dtype)
    return c


def mamba1_prefill_case(seed, new_tokens, num_computed, Dc, N, G, chunk_size, dtype=torch.bfloat16, device="cpu",
                        has_init=None, num_slots=None, null_block_id=0, gate=False):
    """A varlen Mamba1 prefill batch ("all" cache mode): x, dt [T, Dc], B, C [T, G, N], A [Dc, N],
    D and dt_bias [Dc], cache [slots, Dc, N] (sentinel except the slots read as initial states)."""
    c = prefill_case(seed, new_tokens, num_computed, Dc, 1, N, G, chunk_size, dtype=dtype, device=device,
                     has_init=has_init, num_slots=num_slots, null_block_id=null_block_id, mode="all")
    return _as_mamba1(c, N, seed, device, gate)


def mamba1_decode_case(seed, live, padded, tokens_per_req, Dc, N, G, num_slots, dtype=torch.bfloat16,
                       device="cpu", null_block_id=0, gate=False):
    """A padded Mamba1 decode batch, routed as decode_case."""
    c = decode_case(seed, live, padded, tokens_per_req, Dc, 1, N, G, num_slots, dtype=dtype, device=device,
                    null_block_id=null_block_id)
    return _as_mamba1(c, N, seed, device, gate)
