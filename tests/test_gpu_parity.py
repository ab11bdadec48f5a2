"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
identical seeded bf16 inputs, at sizes the oracle finishes in seconds that
still span several 128-row tiles and a ragged tail.

Bar: kept-block bitmaps bit-exact (thresholds and ln(lambda) guarded clear of
every compared value by >= 1e-3); outputs within max-abs 2e-2 and mean-abs
2e-3; log-sum-exp within 2e-3."""
import math

import numpy as np
import pytest
import torch

from block_sparse_gated_gb300 import workloads as wl
from oracle import bsfa_oracle as orc
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _bsfa():
    import block_sparse_gated_gb300 as b
    return b


def _inputs(Hq, Hkv, L, d, seed, dev, **kw):
    x = wl.layer_inputs(Hq, Hkv, L, d, seed, device="cpu", **kw)
    return x, x.q.to(dev), x.k.to(dev), x.v.to(dev)


# Gated 128 x 128 calls run the one-head kernel by default ("auto"); the
# cases below that take `schedule` also run the paired kernel explicitly.
SCHEDULES = ["auto", "paired"]


def _skip_redundant(schedule, Bq=128, Bk=128):
    if schedule == "paired" and (Bq, Bk) != (128, 128):
        pytest.skip("auto already runs the paired kernel for these block sizes")


def _run(q, k, v, **kw):
    b = _bsfa()
    r = b.prefill(q[None], k[None], v[None], return_bitmap=True, return_lse=True,
                  return_counts=True, **kw)
    torch.cuda.synchronize()
    assert b.api.device_error() == 0
    return r


# ---------------------------------------------------------------- dense path
@pytest.mark.parametrize("Hq,Hkv,L,d", [
    (2, 1, 128, 128), (4, 2, 300, 128), (2, 2, 200, 64), (1, 1, 129, 128), (8, 2, 1000, 128),
    (3, 1, 257, 64)])
def test_dense_mode_matches_oracle(cuda_device, Hq, Hkv, L, d):
    x, q, k, v = _inputs(Hq, Hkv, L, d, 11, cuda_device)
    r = _run(q, k, v, mode="none")
    ref = orc.prefill(gu.to64(x.q), gu.to64(x.k), gu.to64(x.v), Bq=128, Bk=128, mode="dense")
    gu.assert_close(gu.to64(r["out"][0]), ref["out"], "out")
    gu.assert_close(gu.to64(r["lse"]).reshape(Hq, L), ref["lse"], "lse", max_abs=gu.LSE_ABS,
                    mean_abs=gu.LSE_ABS)


def test_zero_queries_average_values(cuda_device):
    """Q = 0: every kept weight is equal, so row r is the mean of V over keys
    0..r -- isolates the P.V path from Q.K^T."""
    Hq, Hkv, L, d = 2, 1, 300, 128
    x, q, k, v = _inputs(Hq, Hkv, L, d, 12, cuda_device)
    q = torch.zeros_like(q)
    r = _run(q, k, v, mode="none")
    v64 = gu.to64(x.v)[0]
    ref = np.cumsum(v64, axis=0) / np.arange(1, L + 1)[:, None]
    for h in range(Hq):
        gu.assert_close(gu.to64(r["out"][0, h]), ref, "out")


# ------------------------------------------------------------ threshold gate
def _threshold_case(dev, Hq, Hkv, L, d, Bq, Bk, seed, table, needles=0, sink=0,
                    schedule="auto"):
    x, q, k, v = _inputs(Hq, Hkv, L, d, seed, dev, needles=needles, sink_tokens=sink,
                         block=max(Bq, Bk))
    q64, k64, v64 = gu.to64(x.q), gu.to64(x.k), gu.to64(x.v)
    sigma = gu.default_sigma(d)
    T, n_adj, _ = gu.guarded_thresholds(q64, k64, table, Bq, Bk, sigma)
    r = _run(q, k, v, block_q=Bq, block_k=Bk, mode="threshold",
             thresholds=torch.from_numpy(T).to(dev), schedule=schedule)
    ref = orc.prefill(q64, k64, v64, Bq=Bq, Bk=Bk, thresholds=T.astype(np.float64))
    bits, clean = gu.unpack_bitmap(r["bitmap"], Hq, [L], Bq, Bk)
    assert clean
    mism = np.argwhere(bits[0] != ref["keep"])
    assert mism.size == 0, f"{len(mism)} bitmap mismatches, first {mism[:5].tolist()}"
    gu.assert_close(gu.to64(r["out"][0]), ref["out"], "out")
    gu.assert_close(gu.to64(r["lse"]).reshape(Hq, L), ref["lse"], "lse", max_abs=gu.LSE_ABS,
                    mean_abs=gu.LSE_ABS)
    cnt = r["counts"].cpu().tolist()
    cand = ref["candidate"]
    assert cnt[0] == int((ref["keep"] & cand).sum())
    assert cnt[1] == int(cand.sum())
    assert cnt[2] == int((ref["visible"] & ~cand).sum())
    return ref


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("Bq,Bk", [(128, 128), (64, 64), (128, 64), (64, 128)])
@pytest.mark.parametrize("Hq,Hkv,L,d", [(4, 2, 1000, 128), (2, 2, 700, 64), (4, 1, 513, 128)])
def test_threshold_gate_matches_oracle(cuda_device, Bq, Bk, Hq, Hkv, L, d, schedule):
    _skip_redundant(schedule, Bq, Bk)
    x = wl.layer_inputs(Hq, Hkv, L, d, 21, needles=2, block=max(Bq, Bk))
    table = gu.median_table(gu.to64(x.q), gu.to64(x.k), Bq, Bk, gu.default_sigma(d))
    ref = _threshold_case(cuda_device, Hq, Hkv, L, d, Bq, Bk, 21, table, needles=2,
                          schedule=schedule)
    cand = ref["candidate"]
    kept = (ref["keep"] & cand).sum()
    assert 0 < kept < cand.sum()  # the case really gates


@pytest.mark.parametrize("fill", [-np.inf, np.inf])
def test_threshold_limits(cuda_device, fill):
    Hq, Hkv, L, d = 4, 2, 777, 128
    table = np.full((Hq, 3), fill, dtype=np.float32)
    _threshold_case(cuda_device, Hq, Hkv, L, d, 128, 128, 22, table)


def test_last_position_reuse(cuda_device):
    Hq, Hkv, L, d = 2, 1, 1100, 128
    x = wl.layer_inputs(Hq, Hkv, L, d, 23)
    table = gu.median_table(gu.to64(x.q), gu.to64(x.k), 128, 128, gu.default_sigma(d))[:, :4]
    ref = _threshold_case(cuda_device, Hq, Hkv, L, d, 128, 128, 23, table)  # nT=4 < 9 blocks
    assert (~ref["keep"][:, 4:] & ref["candidate"][:, 4:]).any()


def test_tiny_workload_calibrated(cuda_device):
    """The tiny workload end to end: calibrate k=4 on 4 seeded samples with the
    oracle, guard, then gate on an independent input."""
    cfg = wl.WORKLOADS["tiny-h2-d64-L1024"]
    Hq, Hkv, L, d, Bq, Bk = (cfg[x] for x in ("Hq", "Hkv", "L", "d", "Bq", "Bk"))
    cal = [wl.layer_inputs(Hq, Hkv, L, d, wl.cal_seed(cfg["index"], n), with_v=False,
                           needles=cfg["cal_needles"], block=Bk) for n in range(cfg["n_cal"])]
    T = orc.calibrate([gu.to64(c.q) for c in cal], [gu.to64(c.k) for c in cal], Bq=Bq, Bk=Bk,
                      ks=cfg["ks"])[0].astype(np.float32)
    ref = _threshold_case(cuda_device, Hq, Hkv, L, d, Bq, Bk, wl.eval_seed(cfg["index"]), T,
                          needles=cfg["needles"])
    assert ref["keep"][:, 4:][ref["candidate"][:, 4:]].any()


# ---------------------------------------------------------------- lambda gate
@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("Bq,Bk,skip_rate", [(128, 128, 0.5), (64, 64, 0.5), (128, 64, 0.5),
                                             (64, 128, 0.5), (128, 128, 0.0)])
def test_lambda_gate_matches_oracle(cuda_device, Bq, Bk, skip_rate, schedule):
    _skip_redundant(schedule, Bq, Bk)
    Hq, Hkv, L, d = 4, 2, 1500, 128
    x, q, k, v = _inputs(Hq, Hkv, L, d, 31, cuda_device, skip_rate=skip_rate, block=Bk)
    q64, k64, v64 = gu.to64(x.q), gu.to64(x.k), gu.to64(x.v)
    sigma = gu.default_sigma(d)
    ll = gu.guarded_log_lambda(-1.0 if skip_rate > 0 else -1e30, Bq, Bk, sigma, [(q64, k64)])
    r = _run(q, k, v, block_q=Bq, block_k=Bk, mode="lambda", log_lambda=ll, schedule=schedule)
    ref = orc.prefill(q64, k64, v64, Bq=Bq, Bk=Bk, mode="lambda", log_lambda=ll)
    bits, clean = gu.unpack_bitmap(r["bitmap"], Hq, [L], Bq, Bk)
    assert clean
    mism = np.argwhere(bits[0] != ref["keep"])
    assert mism.size == 0, f"{len(mism)} bitmap mismatches, first {mism[:5].tolist()}"
    gu.assert_close(gu.to64(r["out"][0]), ref["out"], "out")
    if skip_rate > 0:
        assert (~ref["keep"] & ref["visible"]).any()


# ---------------------------------------------------------------- varlen
@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("mode", ["threshold", "lambda", "none"])
def test_varlen_matches_oracle(cuda_device, mode, schedule):
    if schedule == "paired" and mode == "none":
        pytest.skip("auto already runs the paired kernel with the gate compiled out")
    Hq, Hkv, d, B = 4, 2, 128, 128
    lens = [100, 0, 300, 129, 640, 1]
    parts = [wl.layer_inputs(Hq, Hkv, Ln, d, 40 + n, skip_rate=0.4) if Ln else None
             for n, Ln in enumerate(lens)]
    qs = [p.q if p else torch.empty(Hq, 0, d, dtype=torch.bfloat16) for p in parts]
    ks = [p.k if p else torch.empty(Hkv, 0, d, dtype=torch.bfloat16) for p in parts]
    vs = [p.v if p else torch.empty(Hkv, 0, d, dtype=torch.bfloat16) for p in parts]
    q, cu = wl.pack_varlen(qs)
    k, _ = wl.pack_varlen(ks)
    v, _ = wl.pack_varlen(vs)
    q64, k64, v64 = gu.to64(q), gu.to64(k), gu.to64(v)
    sigma = gu.default_sigma(d)
    kw = {}
    T = None
    if mode == "threshold":
        bounds = [(a, e) for a, e in zip(cu[:-1].tolist(), cu[1:].tolist()) if e > a]
        T = gu.median_table(None, None, B, B, sigma,
                            seq_slices=[(q64[:, a:e], k64[:, a:e]) for a, e in bounds])
        slices = [(q64[:, a:e], k64[:, a:e], [(h, i) for h in range(Hq)
                                               for i in range(orc.num_blocks(e - a, B))])
                  for a, e in bounds]
        T, _, _ = gu.guarded_thresholds(None, None, T, B, B, sigma, seq_slices=slices)
        kw = dict(thresholds=torch.from_numpy(T).to(cuda_device))
    elif mode == "lambda":
        ll = gu.guarded_log_lambda(-1.0, B, B, sigma, gu.varlen_slices(q64, k64, cu.tolist()))
        kw = dict(log_lambda=ll)
    b = _bsfa()
    r = b.prefill(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                  cu_seqlens=cu.to(cuda_device), max_seqlen=max(lens), mode=mode,
                  return_bitmap=True, return_lse=True, schedule=schedule, **kw)
    torch.cuda.synchronize()
    assert b.api.device_error() == 0
    okw = dict(mode={"none": "dense"}.get(mode, mode))
    if mode == "threshold":
        okw["thresholds"] = T.astype(np.float64)
    if mode == "lambda":
        okw["log_lambda"] = ll
    ref = orc.prefill_varlen(q64, k64, v64, cu.numpy(), Bq=B, Bk=B, **okw)
    bits, clean = gu.unpack_bitmap(r["bitmap"], Hq, lens, B, B)
    assert clean
    for n, Ln in enumerate(lens):
        if Ln:
            assert np.array_equal(bits[n], ref["keep"][n]), f"sequence {n}"
    gu.assert_close(gu.to64(r["out"]), ref["out"], "out")
    gu.assert_close(gu.to64(r["lse"]), ref["lse"], "lse", max_abs=gu.LSE_ABS, mean_abs=gu.LSE_ABS)


# ---------------------------------------------------------------- layouts
def test_blhd_layout_matches_bhld(cuda_device):
    Hq, Hkv, L, d = 4, 2, 400, 128
    x, q, k, v = _inputs(Hq, Hkv, L, d, 51, cuda_device)
    b = _bsfa()
    a = b.prefill(q[None], k[None], v[None], mode="none")["out"]
    qt, kt, vt = (t[None].transpose(1, 2).contiguous() for t in (q, k, v))
    o = b.prefill(qt, kt, vt, mode="none", layout="blhd")["out"]
    torch.cuda.synchronize()
    assert torch.equal(o.transpose(1, 2), a)


def test_batch_of_two_matches_single_calls(cuda_device):
    Hq, Hkv, L, d = 4, 2, 333, 128
    xs = [wl.layer_inputs(Hq, Hkv, L, d, 60 + n) for n in range(2)]
    b = _bsfa()
    q = torch.stack([x.q for x in xs]).to(cuda_device)
    k = torch.stack([x.k for x in xs]).to(cuda_device)
    v = torch.stack([x.v for x in xs]).to(cuda_device)
    both = b.prefill(q, k, v, mode="lambda", log_lambda=-2.0)["out"]
    for n in range(2):
        one = b.prefill(q[n:n + 1], k[n:n + 1], v[n:n + 1], mode="lambda", log_lambda=-2.0)["out"]
        torch.cuda.synchronize()
        assert torch.equal(one[0], both[n])


# ---------------------------------------------------------------- calibration
@pytest.mark.parametrize("Bq,Bk,d,Hq,Hkv", [(128, 128, 128, 4, 2), (64, 64, 64, 2, 2),
                                            (128, 64, 128, 2, 1), (64, 128, 128, 4, 1)])
def test_calibrate_matches_oracle(cuda_device, Bq, Bk, d, Hq, Hkv):
    L, N, ks = 1100, 3, [1, 3, 8]
    sam = [wl.layer_inputs(Hq, Hkv, L, d, 70 + n, with_v=False, needles=2, block=Bk)
           for n in range(N)]
    b = _bsfa()
    T = b.calibrate([s.q.to(cuda_device) for s in sam], [s.k.to(cuda_device) for s in sam], ks,
                    block_q=Bq, block_k=Bk)
    torch.cuda.synchronize()
    assert b.api.device_error() == 0
    ref = orc.calibrate([gu.to64(s.q) for s in sam], [gu.to64(s.k) for s in sam], Bq=Bq, Bk=Bk,
                        ks=ks)
    got = T.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref))
    fin = np.isfinite(ref)
    assert np.max(np.abs(got[fin] - ref[fin])) < 1e-4


def test_soak_back_to_back_launches(cuda_device):
    """Many back-to-back launches give the same bitmap and output bytes."""
    Hq, Hkv, L, d = 8, 2, 2048, 128
    x, q, k, v = _inputs(Hq, Hkv, L, d, 81, cuda_device, skip_rate=0.5)
    b = _bsfa()
    first = b.prefill(q[None], k[None], v[None], mode="lambda", log_lambda=-1.0,
                      return_bitmap=True)
    outs = [b.prefill(q[None], k[None], v[None], mode="lambda", log_lambda=-1.0,
                      return_bitmap=True) for _ in range(50)]
    torch.cuda.synchronize()
    assert b.api.device_error() == 0
    for o in outs:
        assert torch.equal(o["out"], first["out"])
        assert torch.equal(o["bitmap"], first["bitmap"])


# ------------------------------------------------------- V loaded for every tile
@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("mode", ["threshold", "lambda"])
@pytest.mark.parametrize("Bq,Bk,d", [(128, 128, 128), (64, 64, 64)])
def test_v_always_is_bit_identical(cuda_device, mode, Bq, Bk, d, schedule):
    _skip_redundant(schedule, Bq, Bk)
    """Loading V for skipped tiles too (the flag that exists for the A/B
    against skipping the load) changes no output bit; the case does skip
    blocks."""
    Hq, Hkv, L = 4, 2, 1500
    x, q, k, v = _inputs(Hq, Hkv, L, d, 91, cuda_device, skip_rate=0.6, needles=2, block=Bk)
    kw = dict(block_q=Bq, block_k=Bk, mode=mode, schedule=schedule)
    if mode == "lambda":
        kw["log_lambda"] = -1.0
    else:
        table = gu.median_table(gu.to64(x.q), gu.to64(x.k), Bq, Bk, gu.default_sigma(d))
        kw["thresholds"] = torch.from_numpy(table.astype(np.float32)).to(cuda_device)
    a = _run(q, k, v, **kw)
    b = _run(q, k, v, v_always=True, **kw)
    assert torch.equal(a["out"], b["out"])
    assert torch.equal(a["bitmap"], b["bitmap"])
    assert torch.equal(a["lse"], b["lse"])
    kept, cand = a["counts"].cpu().tolist()[:2]
    assert 0 < kept < cand


# ------------------------------------------------- gates that keep everything
@pytest.mark.parametrize("schedule", SCHEDULES)
def test_keep_all_gate_with_and_without_vote(cuda_device, schedule):
    """A -inf threshold row (or ln(lambda) = -inf) keeps every block without
    a vote (paired kernel) or without keeping an exact running max (one-head
    kernel); -1e30 keeps every block after a vote.  All give the same bytes."""
    Hq, Hkv, L, d = 4, 2, 1000, 128
    x, q, k, v = _inputs(Hq, Hkv, L, d, 95, cuda_device, skip_rate=0.5)
    s = dict(schedule=schedule)
    a = _run(q, k, v, mode="threshold", thresholds=torch.full((Hq, 1), -math.inf, device=cuda_device), **s)
    b = _run(q, k, v, mode="threshold", thresholds=torch.full((Hq, 1), -1e30, device=cuda_device), **s)
    c = _run(q, k, v, mode="lambda", log_lambda=-math.inf, **s)
    d_ = _run(q, k, v, mode="lambda", log_lambda=-1e30, **s)
    for r in (b, c, d_):
        for key in ("out", "lse", "bitmap", "counts"):
            assert torch.equal(a[key], r[key]), key
    kept, cand = a["counts"].cpu().tolist()[:2]
    assert kept == cand


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_mixed_trivial_and_voting_units(cuda_device, schedule):
    """Within one call, units whose threshold entries are all -inf (no vote)
    next to units that vote, including the two query heads of one CTA (a
    GQA pair) taking different paths: against the oracle."""
    Hq, Hkv, L, d = 4, 2, 1300, 128
    x = wl.layer_inputs(Hq, Hkv, L, d, 96, needles=2)
    table = gu.median_table(gu.to64(x.q), gu.to64(x.k), 128, 128, gu.default_sigma(d))
    table[0, ::2] = -np.inf        # head 0: every other query block without a vote
    table[2, :] = -np.inf          # head 2: all -inf, its pair partner (head 3) votes
    table[1, 5:] = -np.inf         # head 1: -inf from query block 5 on
    ref = _threshold_case(cuda_device, Hq, Hkv, L, d, 128, 128, 96, table, needles=2,
                          schedule=schedule)
    cand = ref["candidate"]
    assert (ref["keep"][3] & cand[3]).sum() < cand[3].sum()  # head 3 really gates


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_high_skip_soak_many_units_per_cta(cuda_device, schedule):
    """About 94% of the candidates skipped, query blocks below the budget at
    -inf (kept without a vote), many units per CTA, 20 back-to-back calls:
    no bounded wait may run out (a softmax running through skipped tiles
    ahead of the V loader must not confuse its decision reads), and every
    call gives the same bytes."""
    Hq, Hkv, L, d, kb = 32, 8, 16384, 128, 8
    x, q, k, v = _inputs(Hq, Hkv, L, d, 97, cuda_device, needles=4, block=128)
    b = _bsfa()
    nq = L // 128
    # Per-row budget kb from the oracle's block maxima of two heads; the
    # other heads take the median of those rows (the schedule does not care
    # which heads the values come from).
    q64, k64 = gu.to64(x.q), gu.to64(x.k)
    sigma = gu.default_sigma(d)
    T = np.full((Hq, nq), -np.inf, dtype=np.float32)
    for h in (0, 17):
        sm = orc.block_maxima(q64[h], k64[h // 4], 128, 128, sigma)
        for i in range(kb, nq):
            T[h, i] = orc.kth_largest(list(sm[i][np.isfinite(sm[i])]), kb)
    fill = np.median(T[[0, 17]][:, kb:])
    T[:, kb:] = np.where(np.isfinite(T[:, kb:]), T[:, kb:], fill)
    Td = torch.from_numpy(T).to(cuda_device)
    first = b.prefill(q[None], k[None], v[None], mode="threshold", thresholds=Td,
                      return_bitmap=True, return_counts=True, schedule=schedule)
    torch.cuda.synchronize()
    assert b.api.device_error() == 0
    kept, cand = first["counts"].cpu().tolist()[:2]
    assert 1 - kept / cand > 0.85
    for _ in range(20):
        r = b.prefill(q[None], k[None], v[None], mode="threshold", thresholds=Td,
                      return_bitmap=True, schedule=schedule)
        torch.cuda.synchronize()
        assert b.api.device_error() == 0
        assert torch.equal(r["out"], first["out"])
        assert torch.equal(r["bitmap"], first["bitmap"])
