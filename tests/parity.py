"""Shared parity helpers: run the CUDA path on a seeded case and compare it
with the CPU oracle on the same (bf16-rounded) inputs.

Tolerance, as a ratio max|gpu - oracle| / RMS(oracle) over the compared
elements: 2e-2 for bf16 inputs and 1e-4 for fp32 inputs.  States are fp32
and are compared that way.  y is stored in the input dtype; for bf16 that
storage alone moves a value by up to half a bf16 ulp, which for these
heavy-tailed outputs (max|y| / RMS(y) reaches 40) exceeds 2e-2 of the RMS
even for the exactly rounded oracle.  So for bf16 y the error counted is the
part beyond half an ulp at the element's magnitude: it bounds the error of
the value the kernel computed before it was stored.  Slot ids, chunk metadata
and slots the call must not touch are compared bit for bit.
"""
import math

import numpy as np
import torch

import oracle
import selective_state_space_mamba2_gb300 as ssd

TOL = {torch.bfloat16: 2e-2, torch.float32: 1e-4}


def rel_err(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    if a.size == 0:
        return 0.0
    rms = math.sqrt(float(np.mean(b * b)))
    return float(np.max(np.abs(a - b))) / max(rms, 1e-30)


def ulp_bf16(v):
    """Spacing of bf16 numbers at magnitude |v| (8 significant bits)."""
    a = np.maximum(np.abs(np.asarray(v, np.float64)), 1.1754943508222875e-38)
    return np.exp2(np.floor(np.log2(a)) - 7)


def y_err(got, want, dtype):
    """max error / RMS(want); for bf16 outputs the first half ulp is excused."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    if got.size == 0:
        return 0.0
    if dtype != torch.bfloat16:
        return rel_err(got, want)
    allow = 0.5 * ulp_bf16(np.maximum(np.abs(got), np.abs(want)))
    excess = np.maximum(np.abs(got - want) - allow, 0.0)
    rms = math.sqrt(float(np.mean(want * want)))
    return float(excess.max()) / max(rms, 1e-30)


def y_err_pair(a, b, dtype):
    """Like y_err, for two outputs of the GPU path: when both were rounded to
    bf16, each rounding moves a value by up to half an ulp, so one ulp is
    excused; normalised by RMS(b)."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    if a.size == 0:
        return 0.0
    if dtype != torch.bfloat16:
        return rel_err(a, b)
    allow = ulp_bf16(np.maximum(np.abs(a), np.abs(b)))
    excess = np.maximum(np.abs(a - b) - allow, 0.0)
    return float(excess.max()) / max(math.sqrt(float(np.mean(b * b))), 1e-30)


def where_worst(got, want, meta=None):
    """Short description of where |got - want| is largest (for failure messages)."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    d = np.abs(got - want)
    idx = np.unravel_index(int(np.argmax(d)), d.shape)
    msg = "max at %s: got %.4g want %.4g" % (tuple(int(i) for i in idx), got[idx], want[idx])
    if d.ndim == 3:  # [T, H, P]: worst tokens and heads
        per_t = d.max(axis=(1, 2))
        bad_t = np.nonzero(per_t > 0.02 * max(np.sqrt(np.mean(want * want)), 1e-30))[0]
        msg += "; %d bad tokens %s" % (len(bad_t), bad_t[:12].tolist())
        per_h = d.max(axis=(0, 2))
        msg += "; per-head max %s" % np.round(per_h, 3).tolist()[:8]
        if meta is not None and len(bad_t):
            cc = np.asarray(meta["cu_chunk_seqlens"])
            ks = np.searchsorted(cc, bad_t, side="right") - 1
            msg += "; chunks %s offsets %s" % (sorted(set(ks.tolist()))[:8],
                                               sorted(set((bad_t - cc[ks]).tolist()))[:12])
    return msg


def prefill_metadata(case):
    return ssd.ssd_chunk_metadata(case["cu_seqlens"], case["chunk_size"], case["num_computed"],
                                  case["has_init"], block_table=case["block_table"],
                                  state_indices=case["state_indices"],
                                  null_block_id=case["null_block_id"])


def run_prefill(case, meta=None, err=None, **kw):
    """Runs ssd_prefill_varlen on the case's device tensors.  Returns (y, meta)."""
    dev = case["x"].device
    meta = meta or prefill_metadata(case)
    t = {k: torch.from_numpy(v).to(dev) for k, v in meta.items()}
    y = ssd.ssd_prefill_varlen(
        case["x"], case["dt"], case["A"], case["B"], case["C"], case["cu_seqlens"].to(dev),
        t["cu_chunk_seqlens"], t["seq_idx"], t["last_chunk_indices"], init_slot=t["init_slot"],
        chunk_slot=t["chunk_slot"], state_cache=case["cache"], D=kw.pop("D", case["D"]),
        dt_bias=kw.pop("dt_bias", case["dt_bias"]), null_block_id=case["null_block_id"],
        chunk_size=case["chunk_size"], err_word=err, seq_order=t.get("seq_order"), **kw)
    return y, meta


def _head_subset(case, heads):
    H = case["x"].shape[1]
    G = case["B"].shape[1]
    grp = [h // (H // G) for h in heads]
    return grp


def oracle_prefill(case, meta, cache_before, heads=None, D="case", dt_bias="case",
                   dt_limit=(0.0, math.inf), dt_softplus=True, z=None):
    """fp64 oracle on all heads, or on ``heads`` only (each with its group's
    B/C, as an independent one-head-per-group problem).  Returns
    (y [T,h,P], chunk_states [K,h,P,N])."""
    x, dt, B, C = case["x"], case["dt"], case["B"], case["C"]
    A = case["A"]
    Dv = case["D"] if isinstance(D, str) else D
    bv = case["dt_bias"] if isinstance(dt_bias, str) else dt_bias
    if heads is not None:
        grp = _head_subset(case, heads)
        hs = torch.tensor(heads)
        gs = torch.tensor(grp)
        x, dt = x[:, hs], dt[:, hs]
        B, C = B[:, gs], C[:, gs]
        A = A[hs]
        z = None if z is None else z[:, hs]
        Dv = None if Dv is None else Dv[hs]
        bv = None if bv is None else bv[hs]
    S = len(meta["init_slot"])
    Hs = x.shape[1]
    P, N = x.shape[2], B.shape[2]
    init = np.zeros((S, Hs, P, N))
    has = np.zeros(S, bool)
    null = case["null_block_id"]
    for r in range(S):
        s = int(meta["init_slot"][r])
        if s != null:
            st = cache_before[s]
            if heads is not None:
                st = st[torch.tensor(heads)]
            init[r] = st.double().cpu().numpy()
            has[r] = True
    y, cs, _ = oracle.ssd_prefill(x.cpu(), dt.cpu(), A.cpu(), B.cpu(), C.cpu(), case["cu_seqlens"],
                                  meta["cu_chunk_seqlens"], D=None if Dv is None else Dv.cpu(),
                                  dt_bias=None if bv is None else bv.cpu(), initial_states=init,
                                  has_initial_states=has, dt_softplus=dt_softplus, dt_limit=dt_limit,
                                  z=None if z is None else z.cpu())
    return y, cs


def check_prefill(case, y_gpu, meta, cache_before, cache_after, heads=None, **okw):
    """Compares y and every stored chunk state (sampled heads or all) with the
    oracle, and checks that slots no chunk writes are bit-identical."""
    tol = TOL[case["x"].dtype]
    yo, cso = oracle_prefill(case, meta, cache_before, heads=heads, **okw)
    hs = slice(None) if heads is None else torch.tensor(heads)
    yg = y_gpu[:, hs].double().cpu().numpy()
    e_y = y_err(yg, yo, case["x"].dtype)
    if e_y > tol:
        print("y mismatch:", where_worst(yg, yo, meta))
    null = case["null_block_id"]
    written = [(k, int(s)) for k, s in enumerate(meta["chunk_slot"]) if int(s) != null]
    e_s = 0.0
    if written:
        ks = [k for k, _ in written]
        sl = torch.tensor([s for _, s in written], device=cache_after.device)
        got = cache_after[sl][:, hs].double().cpu().numpy()
        e_s = rel_err(got, cso[ks])
        if e_s > tol:
            print("state mismatch:", where_worst(got, cso[ks]))
    # untouched slots: bitwise
    mask = torch.ones(cache_after.shape[0], dtype=torch.bool, device=cache_after.device)
    if written:
        mask[torch.tensor([s for _, s in written], device=cache_after.device)] = False
    same = torch.equal(cache_after[mask].view(torch.int32), cache_before[mask].view(torch.int32))
    return e_y, e_s, same, tol


def run_decode(case, err=None, **kw):
    dev = case["x"].device
    na = case["num_accepted"]
    y = torch.full_like(case["x"], float("nan"))
    ssd.ssm_decode_update(case["x"], case["dt"], case["A"], case["B"], case["C"], case["cache"],
                          case["state_indices"].to(dev), None if na is None else na.to(dev), out=y,
                          D=case["D"], dt_bias=case["dt_bias"], null_block_id=case["null_block_id"],
                          err_word=err, **kw)
    return y


def check_decode(case, y_gpu, cache_before, cache_after, requests=None, check_untouched=True, z=None):
    """Oracle decode for ``requests`` (all rows if None): y, every written
    state, padded rows untouched, and every slot no live request writes
    bit-identical."""
    tol = TOL[case["x"].dtype]
    si = case["state_indices"].numpy()
    na = case["num_accepted"]
    na = None if na is None else na.numpy()
    null = case["null_block_id"]
    R = si.shape[0]
    tpr = case["tokens_per_req"]
    req = list(range(R)) if requests is None else list(requests)
    rows = torch.tensor([r * tpr + k for r in req for k in range(tpr)])
    rd = oracle.decode_read_slots(si, na, null)
    live = [r for r in req if rd[r] != null]
    read = np.zeros((len(req),) + tuple(cache_after.shape[1:]))
    for i, r in enumerate(req):
        if rd[r] != null:
            read[i] = cache_before[int(rd[r])].double().cpu().numpy()
    yo, st = oracle.ssm_decode(case["x"][rows].cpu(), case["dt"][rows].cpu(), case["A"].cpu(),
                               case["B"][rows].cpu(), case["C"][rows].cpu(), read,
                               [rd[r] != null for r in req], D=case["D"].cpu(),
                               dt_bias=case["dt_bias"].cpu(), z=None if z is None else z[rows].cpu())
    yg = y_gpu[rows].double().cpu().numpy()
    liverows = np.array([rd[r] != null for r in req for _ in range(tpr)])
    e_y = y_err(yg[liverows], yo[liverows], case["x"].dtype)
    dead_ok = bool(np.all(np.isnan(yg[~liverows]))) if (~liverows).any() else True
    got, want = [], []
    for i, r in enumerate(req):
        if rd[r] == null:
            continue
        for k in range(tpr):
            if si[r, k] != null:
                got.append(cache_after[int(si[r, k])].double().cpu().numpy())
                want.append(st[i, k])
    e_s = rel_err(np.stack(got), np.stack(want)) if got else 0.0
    if not check_untouched:
        return e_y, e_s, dead_ok, tol, len(live)
    # slots written by any live request (sampled or not)
    written = set()
    for r in range(R):
        if rd[r] != null:
            written.update(int(s) for s in si[r, :tpr] if s != null)
    mask = torch.ones(cache_after.shape[0], dtype=torch.bool, device=cache_after.device)
    if written:
        mask[torch.tensor(sorted(written), device=cache_after.device)] = False
    same = torch.equal(cache_after[mask].view(torch.int32), cache_before[mask].view(torch.int32))
    return e_y, e_s, same and dead_ok, tol, len(live)


def slot_fingerprints(cache, block=256):
    """Per-slot 64-bit fingerprint of the raw bits (chunked, so no full copy)."""
    S = cache.shape[0]
    out = torch.empty(S, dtype=torch.int64, device=cache.device)
    flat = cache.view(S, -1).view(torch.int32)
    n = flat.shape[1]
    w = (torch.arange(n, device=cache.device, dtype=torch.int64) % 1000003) * 2 + 1
    for a in range(0, S, block):
        b = min(a + block, S)
        out[a:b] = (flat[a:b].to(torch.int64) * w).sum(dim=1)
    return out
