"""Kernel-level parity of the CUDA path (through the C ABI) with the oracle,
on seeded inputs that span several tiles and ragged tails, plus edge cases."""
import math

import numpy as np
import pytest
import torch

from oracle import accept as oaccept
from oracle import fp8 as ofp8
from oracle import indexer as oindexer
from oracle import merge as omerge
from oracle import mla as omla
from oracle import share as oshare
from oracle import topk as otopk
from oracle import writeback as owb

import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mtp_speculative_decode_gb300 as m
    from mtp_speculative_decode_gb300 import _native
    _native.lib()   # raises if the library is missing: no fallback
    return m


def dev(x, dtype=None):
    t = torch.as_tensor(x)
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda().contiguous()


def u32(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.uint32)).cuda()


# ----------------------------------------------------------------------------- merge

@pytest.mark.parametrize("B,K,maxlen", [(1, 0, 3), (2, 3, 2), (37, 5, 4), (300, 5, 1), (5, 2, 0)])
def test_merge(mt, B, K, maxlen):
    rng = np.random.default_rng(B * 10 + K)
    lens = rng.integers(0, maxlen + 1, B)
    po = np.concatenate([[0], np.cumsum(lens)]).astype(np.uint32)
    prompt = rng.integers(0, 10 ** 6, int(po[-1]))
    draft = rng.integers(0, 10 ** 6, (B, K))
    toks, mo = mt.merge_tokens(dev(prompt, torch.int64), u32(po), dev(draft, torch.int64).reshape(B, K))
    want_t, want_o = omerge.merge_tokens(prompt, po, draft)
    assert np.array_equal(toks.cpu().numpy(), want_t)
    assert np.array_equal(mo.cpu().numpy().astype(np.int64), want_o.astype(np.int64))
    assert np.array_equal(mt.host_merged_offsets(po, K), want_o)


# ----------------------------------------------------------------------------- FP8

def test_quantize_bit_exact(mt):
    rng = np.random.default_rng(1)
    x = rng.normal(0, 1, (700, 128)).astype(np.float32)
    x[3] = 0.0
    x[4] = -0.0
    x[5] *= 1e30
    x[6] *= 1e-30
    x[7, :] = 0.0
    x[7, 17] = -2.5
    x[8] = rng.integers(-3, 4, 128).astype(np.float32)    # exact ties after scaling
    codes, scales = mt.quantize_fp8_block128(dev(x))
    want_c, want_s = ofp8.quantize_block128(x)
    assert np.array_equal(scales.cpu().numpy().reshape(-1).view(np.uint32), want_s.reshape(-1).view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), want_c)


# ----------------------------------------------------------------------------- accept

@pytest.mark.parametrize("K", [0, 1, 5, 7])
def test_accept(mt, K):
    rng = np.random.default_rng(K)
    B = 513
    draft = rng.integers(0, 5, (B, K))
    tgt = rng.integers(0, 5, (B, K + 1))
    tgt[: B // 2, :K] = draft[: B // 2]          # long matches
    if K:
        draft[10] = 42                           # sentinel rows
        tgt[10, :K] = 42
    n, nx = mt.accept_greedy(dev(draft, torch.int64).reshape(B, K), dev(tgt, torch.int64), magic_draft_id=42)
    wn, wx = oaccept.accept_greedy(draft, tgt, magic_draft_id=42)
    assert np.array_equal(n.cpu().numpy(), wn) and np.array_equal(nx.cpu().numpy(), wx)


@pytest.mark.parametrize("B,K,V,noise", [(256, 5, 37, 0.5), (300, 1, 1000, 2.0), (64, 0, 500, 0.5),
                                         (16, 5, 154880, 0.3), (40, 7, 4099, 0.05)])
def test_accept_stochastic_exact(mt, B, K, V, noise):
    """Bit-exact against the oracle: accept counts and drawn tokens."""
    from mtp_speculative_decode_gb300 import workloads
    draft, q, p, ua, us = workloads.stochastic_inputs(B + K + V, B, K, V, noise=noise)
    if K > 0 and B > 3:
        draft[1, 0] = V + 5                   # outside the vocabulary: rejected and flagged
        p[2, 0] = 0.5 * q[2, 0]               # residual without mass: the draw falls back to p
        ua[2, 0] = 0.99
        p[3, K] = 0.0                         # a row with no mass at all (reached if all accepted)
        q[3] = p[3, :K]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    n, nx = mt.accept_stochastic(dev(draft), dev(q), dev(p), dev(ua), dev(us), dev_status=status)
    wn, wx = oaccept.accept_stochastic(draft, q, p, ua, us)
    assert np.array_equal(n.cpu().numpy(), wn)
    assert np.array_equal(nx.cpu().numpy(), wx)
    if K > 0 and B > 3:
        assert status.item() & 1, "an out-of-vocabulary draft must be flagged"
        assert wn[1] == 0 and wn[3] == K


# ----------------------------------------------------------------------------- write-back

@pytest.mark.parametrize("lat_dtype", [torch.bfloat16, torch.float32])
def test_writeback_bytes(mt, lat_dtype):
    rng = np.random.default_rng(3)
    B, Wn, T = 40, 6, 3000
    src_l = torch.randn(B, Wn, 576).to(lat_dtype)
    src_k = torch.from_numpy(rng.integers(0, 256, (B, Wn, 128), dtype=np.uint8))
    src_s = torch.rand(B, Wn)
    dst_l = torch.randn(T, 576).to(lat_dtype)
    dst_k = torch.from_numpy(rng.integers(0, 256, (T, 128), dtype=np.uint8))
    dst_s = torch.rand(T)
    n_acc = rng.integers(0, Wn, B).astype(np.int32)
    n_acc[0], n_acc[1] = 0, Wn - 1
    start = np.arange(B) * 70 + rng.integers(0, 10, B)
    start[-1] = T - 2          # last request runs off the pool end: flagged, rest skipped
    g_l, g_k, g_s = dev(dst_l), dev(dst_k), dev(dst_s)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int64, device="cuda")
    cache_start = np.zeros(B, dtype=np.int64)
    cache_start[1::2] = 3               # pool row = cache_start + position
    pos = start - cache_start
    mt.kv_writeback(dev(src_l), dev(src_k), dev(src_s), dev(n_acc), g_l, g_k, g_s, dev(cache_start),
                    dev(pos, torch.int64), next_pos=nxt, dev_status=status)
    acc = np.minimum(n_acc + 1, Wn)
    acc_in = acc.copy()
    acc_in[-1] = min(acc[-1], T - start[-1])
    wl, wk, ws = owb.kv_writeback(src_l.view(torch.int16 if lat_dtype == torch.bfloat16 else torch.int32).numpy(),
                                  src_k.numpy(), src_s.numpy(), acc_in,
                                  dst_l.view(torch.int16 if lat_dtype == torch.bfloat16 else torch.int32).numpy(),
                                  dst_k.numpy(), dst_s.numpy(), start)
    gl = g_l.cpu().view(torch.int16 if lat_dtype == torch.bfloat16 else torch.int32).numpy()
    assert gl.tobytes() == wl.tobytes()
    assert g_k.cpu().numpy().tobytes() == wk.tobytes()
    assert g_s.cpu().numpy().tobytes() == ws.tobytes()
    assert np.array_equal(nxt.cpu().numpy(), pos + acc)
    assert status.item() & 2, "out-of-pool write must be flagged"


# ----------------------------------------------------------------------------- share gather

def test_share_gather(mt):
    rng = np.random.default_rng(4)
    B, k = 50, 64
    lens = rng.integers(1, 7, B)
    ro = np.concatenate([[0], np.cumsum(lens)]).astype(np.uint32)
    s0 = rng.integers(-1, 5000, (int(ro[-1]), k)).astype(np.int32)
    nacc = (rng.integers(0, 7, B) % lens).astype(np.int32)
    got = mt.topk_share_gather(dev(s0), u32(ro), dev(nacc)).cpu().numpy()
    assert np.array_equal(got, oshare.topk_share_gather(s0, ro, nacc))
    got0 = mt.topk_share_gather(dev(s0), u32(ro), None).cpu().numpy()
    assert np.array_equal(got0, oshare.topk_share_gather(s0, ro, None))
    # the position of the reused row comes back with it
    rpos = rng.integers(0, 10 ** 6, int(ro[-1])).astype(np.int64)
    spos = torch.empty(B, dtype=torch.int64, device="cuda")
    got1 = mt.topk_share_gather(dev(s0), u32(ro), dev(nacc), row_pos=dev(rpos), shared_pos=spos).cpu().numpy()
    assert np.array_equal(got1, oshare.topk_share_gather(s0, ro, nacc))
    assert np.array_equal(spos.cpu().numpy(), rpos[ro[:-1].astype(np.int64) + nacc])
    # a local row beyond the segment is clamped to its last row and flagged
    bad = nacc.copy()
    bad[3] = lens[3] + 2
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = mt.topk_share_gather(dev(s0), u32(ro), dev(bad), dev_status=status).cpu().numpy()
    assert np.array_equal(g[3], s0[ro[4] - 1]) and status.item() & 1


# ----------------------------------------------------------------------------- top-k

@pytest.mark.parametrize("V,k,ties", [(10, 32, False), (32, 32, False), (33, 32, True), (5000, 2048, False),
                                      (8198, 2048, True), (60000, 2048, False), (70000, 2048, True),
                                      (3000, 1, True), (4096, 4096, False), (9000, 4096, True),
                                      # one tail key per thread at 1024 threads, 32768+ equal keys in a row
                                      (33000, 2048, True), (37000, 2048, True), (33000, 2048, False),
                                      # split rows: 16384-key segments, then merges of 16384/k lists
                                      (262144, 2048, True), (1048576, 2048, True), (600000, 2048, False),
                                      (1048576, 4096, False), (100000, 7, True), (65536, 2048, True)])
def test_topk_exact(mt, V, k, ties):
    rng = np.random.default_rng(V + k)
    R = 7
    if ties:
        sc = rng.integers(0, 50, (R, V)).astype(np.float32)          # heavy exact ties
        sc[1] = 0.0                                                  # all equal
    else:
        sc = rng.normal(size=(R, V)).astype(np.float32)
    lens = np.full(R, V, dtype=np.int64)
    lens[2] = max(1, V // 3)
    lens[3] = min(V, k)
    lens[4] = 0
    if V > 40960:   # split rows whose last segment holds fewer than k keys
        lens[5] = 16385
        lens[6] = min(V, 2 * 16384 + k - 1)
    ld = V + 4
    buf = np.zeros((R, ld), np.float32)
    buf[:, :V] = sc
    out_s = torch.empty(R, k, dtype=torch.float32, device="cuda")
    got = mt.topk(dev(buf), dev(lens), V, k, out_score=out_s).cpu().numpy()
    gs = out_s.cpu().numpy()
    for r in range(R):
        want = otopk.topk_select(sc[r, :lens[r]].astype(np.float64), k)
        assert np.array_equal(got[r], want.astype(np.int32)), f"row {r}"
        n = min(k, lens[r])
        assert np.array_equal(gs[r, :n], sc[r, got[r, :n]])


def test_topk_split_many_rows(mt):
    """More rows than SMs on the split path (the merge level then runs two CTAs per SM), ragged lengths."""
    rng = np.random.default_rng(11)
    R, V, k = 200, 50000, 2048
    sc = rng.normal(size=(R, V)).astype(np.float32)
    sc[::7] = np.round(sc[::7] * 4)                       # rows with heavy ties
    lens = rng.integers(1, V + 1, R).astype(np.int64)
    lens[0], lens[1], lens[2], lens[3] = V, 40961, k, 16385
    ld = V + 4
    buf = np.zeros((R, ld), np.float32)
    buf[:, :V] = sc
    got = mt.topk(dev(buf), dev(lens), V, k).cpu().numpy()
    for r in range(R):
        want = otopk.topk_select(sc[r, :lens[r]].astype(np.float64), k)
        assert np.array_equal(got[r], want.astype(np.int32)), f"row {r}"


# ----------------------------------------------------------------------------- indexer

def _indexer_case(H, D, lens, r_per, fp8, seed):
    rng = np.random.default_rng(seed)
    B = len(lens)
    cap = np.asarray(lens) + r_per + 3
    cache_start = np.concatenate([[0], np.cumsum(cap)[:-1]]).astype(np.int64)
    T = int(cap.sum())
    row_req = np.repeat(np.arange(B), r_per)
    row_pos = np.repeat(lens, r_per) + np.tile(np.arange(r_per), B)
    R = len(row_req)
    q = rng.normal(size=(R, H, D)).astype(np.float32)
    k = rng.normal(size=(T, D)).astype(np.float32)
    w = rng.uniform(0, 1, (R, H)).astype(np.float32)
    w[0, 0] = -0.5                                   # a negative head weight
    ro = np.concatenate([[0], np.cumsum(np.full(B, r_per))]).astype(np.uint32)
    return dict(q=q, k=k, w=w, cache_start=cache_start, row_req=row_req, row_pos=row_pos, ro=ro, T=T)


@pytest.mark.parametrize("H,D,lens,r_per,k,fp8,split", [
    (4, 64, [100, 300], 4, 32, False, None),                 # the tiny float32 shape
    (64, 128, [300, 1000, 129, 5], 6, 256, True, None),       # several tiles + ragged tails, FP8 (head halves)
    (64, 128, [300, 1000, 129, 5], 6, 256, True, "0"),        # the same without the head halves
    (64, 128, [4100, 200], 1, 2048, True, None),              # draft-step shape: one row per request
    (64, 128, [4100, 200], 1, 2048, True, "1"),               # one row in head halves (N = 32)
    (64, 128, [500, 1300, 129], 5, 512, True, None),          # odd rows: the last pair holds one row
    (64, 128, [700, 64, 2000], 7, 512, True, None),
    (64, 128, [900, 300], 8, 1024, True, None),               # a full pair for warpgroup 0's second unit
    (64, 128, [900, 300, 50], 11, 256, True, None),           # requests cut into groups of 8 + 3 rows
    (32, 128, [777, 1500, 64], 3, 512, True, None),
])
def test_indexer_scores_and_topk(mt, H, D, lens, r_per, k, fp8, split, monkeypatch):
    if split is not None:
        monkeypatch.setenv("MTPSD_INDEXER_SPLIT", split)
    c = _indexer_case(H, D, lens, r_per, fp8, seed=H + D + k)
    R = len(c["row_req"])
    maxv = int(max(c["row_pos"])) + 1
    ld = mt.scores_ld(maxv)
    if fp8:
        qc, qs = ofp8.quantize_block128(c["q"])
        kc, ks = ofp8.quantize_block128(c["k"])
        gq, gqs = mt.quantize_fp8_block128(dev(c["q"]))
        gk, gks = mt.quantize_fp8_block128(dev(c["k"]))
        assert np.array_equal(gq.cpu().numpy(), qc) and np.array_equal(gk.cpu().numpy(), kc)
        qs, ks = qs[..., 0], ks[:, 0]
        gqs, gks = gqs.reshape(R, H).contiguous(), gks.reshape(-1).contiguous()
    else:
        gq, gqs, gk, gks = dev(c["q"]), None, dev(c["k"]), None
    scores = torch.full((R, ld), float("nan"), device="cuda")
    idx = mt.indexer_topk(gq, gqs, dev(c["w"]), gk, gks, dev(c["cache_start"]), u32(c["ro"]),
                          dev(c["row_pos"], torch.int64), k, maxv, scores=scores).cpu().numpy()
    sc = scores.cpu().numpy()
    if fp8:
        ref = oindexer.indexer_scores(qc, qs, c["w"], kc, ks, c["cache_start"], c["row_req"], c["row_pos"], fp8=True)
    else:
        ref = oindexer.indexer_scores(c["q"], None, c["w"], c["k"], None, c["cache_start"], c["row_req"],
                                      c["row_pos"], fp8=False)
    tolerated = 0
    for r in range(R):
        V = int(c["row_pos"][r]) + 1
        parity.check_scores_row(sc[r, :V], ref[r])
        tolerated += parity.check_topk_row(idx[r], ref[r], k)
    print(f"top-k differences inside the tie band: {tolerated}")
    # the two halves called separately (score GEMM, then the standalone top-k over row_pos + 1
    # positions) give exactly the fused call's scores and selection
    gpos = dev(c["row_pos"], torch.int64)
    sc2 = mt.indexer_scores(gq, gqs, dev(c["w"]), gk, gks, dev(c["cache_start"]), u32(c["ro"]), gpos, maxv)
    idx2 = mt.topk(sc2, gpos, maxv, k, row_len_add=1).cpu().numpy()
    sc2 = sc2.cpu().numpy()
    for r in range(R):
        V = int(c["row_pos"][r]) + 1
        assert np.array_equal(sc2[r, :V].view(np.uint32), sc[r, :V].view(np.uint32))
    assert np.array_equal(idx2, idx)


# ----------------------------------------------------------------------------- sparse MLA

def _mla_case(H, lens, n_idx, dtype, seed, n_rows=3):
    rng = np.random.default_rng(seed)
    B = len(lens)
    cap = np.asarray(lens) + 8
    cache_start = np.concatenate([[0], np.cumsum(cap)[:-1]]).astype(np.int64)
    T = int(cap.sum())
    row_req = np.repeat(np.arange(B), n_rows)
    row_pos = np.repeat(lens, n_rows) + np.tile(np.arange(n_rows), B)
    R = len(row_req)
    g = torch.Generator().manual_seed(seed)
    latent = torch.randn(T, 576, generator=g).to(dtype)
    q = torch.randn(R, H, 576, generator=g).to(dtype)
    idx = np.full((R, n_idx), -1, dtype=np.int32)
    for r in range(R):
        V = int(row_pos[r]) + 1
        sel = np.sort(rng.choice(V, size=min(V, n_idx), replace=False))
        idx[r, :len(sel)] = sel
    ro = np.concatenate([[0], np.cumsum(np.full(B, n_rows))]).astype(np.uint32)
    return dict(latent=latent, q=q, idx=idx, cache_start=cache_start, row_req=row_req, row_pos=row_pos, ro=ro)


@pytest.mark.parametrize("H,lens,n_idx,dtype", [
    (8, [100, 300], 32, torch.float32),
    (128, [300, 2100, 50], 512, torch.bfloat16),
    (128, [9000], 2048, torch.bfloat16),
    (16, [700, 40], 256, torch.bfloat16),          # heads below one 64-head group
    (80, [1000, 3000, 5], 1000, torch.bfloat16),   # ragged head group, n_idx not a tile multiple
])
def test_sparse_mla(mt, H, lens, n_idx, dtype):
    c = _mla_case(H, lens, n_idx, dtype, seed=H + n_idx)
    R = len(c["row_req"])
    scale = 1.0 / math.sqrt(576.0)
    lse = torch.empty(R, H, device="cuda")
    out = mt.sparse_mla_decode(dev(c["q"]), dev(c["latent"]), dev(c["cache_start"]), u32(c["ro"]),
                               dev(c["row_pos"], torch.int64), dev(c["idx"]), scale, lse=lse)
    ref = omla.sparse_mla(c["q"], c["latent"], c["cache_start"], c["row_req"], c["idx"], scale)
    tol = parity.ATT_TOL_F32 if dtype == torch.float32 else parity.ATT_TOL_BF16
    o = out.float().cpu().numpy()
    ls = lse.cpu().numpy()
    worst = 0.0
    for r in range(R):
        worst = max(worst, parity.check_attention_row(o[r], ref[r][0], tol))
        assert np.max(np.abs(ls[r] - ref[r][1])) <= (1e-4 if dtype == torch.float32 else 2e-3) * max(
            1.0, np.max(np.abs(ref[r][1])))
    print(f"worst relative L2 error {worst:.2e}")


@pytest.mark.parametrize("H,lens,n_idx,n_rows,n_append,force", [
    (128, [300, 2100, 50], 512, 3, 0, True),      # one pair per cluster: every row in 8 pieces, masked pieces
    (128, [9000], 2048, 3, 0, True),              # 16 pieces per row
    (256, [700, 40], 256, 2, 0, True),            # two head groups per row
    (128, [5000, 64], 2048, 2, 1, True),          # an appended position: a last pair of one position
    (128, [3000] * 30, 256, 3, 0, False),         # 90 rows: the default choice, whole rows and cut ones
    (128, [1200] * 40, 128, 2, 2, False),         # 80 rows, two pairs each with appended positions
])
def test_sparse_mla_persistent(mt, H, lens, n_idx, n_rows, n_append, force, monkeypatch):
    """The persistent launch: clusters take equal runs of pairs across rows, and rows cut between
    clusters are merged from their pieces."""
    if force:
        monkeypatch.setenv("MTPSD_MLA_PERSIST", "1")
    c = _mla_case(H, lens, n_idx, torch.bfloat16, seed=H + n_idx + n_rows, n_rows=n_rows)
    R = len(c["row_req"])
    scale = 1.0 / math.sqrt(576.0)
    base = c["row_pos"].astype(np.int64) - n_append
    idx = c["idx"].copy()
    idx[idx > base[:, None]] = -1
    lse = torch.empty(R, H, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = mt.sparse_mla_decode(dev(c["q"]), dev(c["latent"]), dev(c["cache_start"]), u32(c["ro"]),
                               dev(base, torch.int64), dev(idx), scale, n_append=n_append,
                               append_base=dev(base, torch.int64) if n_append else None, row_pos_add=n_append,
                               lse=lse, dev_status=status)
    assert status.item() == 0
    ref = omla.sparse_mla(c["q"], c["latent"], c["cache_start"], c["row_req"], idx, scale, n_append=n_append,
                          append_base=base if n_append else None)
    o = out.float().cpu().numpy()
    ls = lse.cpu().numpy()
    worst = 0.0
    for r in range(R):
        worst = max(worst, parity.check_attention_row(o[r], ref[r][0], parity.ATT_TOL_BF16))
        assert np.max(np.abs(ls[r] - ref[r][1])) <= 2e-3 * max(1.0, np.max(np.abs(ref[r][1])))
    # the same call on the split launch gives the same rows within the tolerance
    monkeypatch.setenv("MTPSD_MLA_PERSIST", "0")
    out0 = mt.sparse_mla_decode(dev(c["q"]), dev(c["latent"]), dev(c["cache_start"]), u32(c["ro"]),
                                dev(base, torch.int64), dev(idx), scale, n_append=n_append,
                                append_base=dev(base, torch.int64) if n_append else None, row_pos_add=n_append)
    o0 = out0.float().cpu().numpy()
    for r in range(R):
        parity.check_attention_row(o[r], o0[r].astype(np.float64), parity.ATT_TOL_BF16)
    print(f"worst relative L2 error {worst:.2e}")


# ----------------------------------------------------------------------------- FP8 latent cache

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_pack_latent_fp8_bit_exact(mt, dtype):
    g = torch.Generator().manual_seed(17)
    x = torch.randn(1500, 576, generator=g).to(dtype)
    x[3] = 0
    x[4, :128] = 0                                   # a block without mass: scale 1
    x[5] *= 1e3
    got = mt.pack_latent_fp8(dev(x)).cpu().numpy()
    want = omla.pack_fp8_ds_mla(x.float().numpy())
    assert got.tobytes() == want.tobytes()


@pytest.mark.parametrize("H,lens,n_idx,n_append", [
    (128, [300, 2100, 50], 512, 0),
    (128, [9000], 2048, 0),                           # several splits, merged
    (64, [700, 40], 256, 3),                          # appended positions, a row shorter than n_idx
    (128, [5000, 64], 2048, 1),
])
def test_sparse_mla_fp8_latent(mt, H, lens, n_idx, n_append):
    """Sparse MLA over the 656-byte FP8 latent rows against the oracle over their exact dequantization."""
    c = _mla_case(H, lens, n_idx, torch.bfloat16, seed=H + n_idx + 5)
    R = len(c["row_req"])
    scale = 1.0 / math.sqrt(576.0)
    packed = mt.pack_latent_fp8(dev(c["latent"]))
    lat_deq = omla.unpack_fp8_ds_mla(omla.pack_fp8_ds_mla(c["latent"].float().numpy()))
    base = c["row_pos"].astype(np.int64) - n_append
    idx = c["idx"].copy()
    idx[idx > base[:, None]] = -1                     # the selection sees positions up to base
    lse = torch.empty(R, H, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = mt.sparse_mla_decode(dev(c["q"]), packed, dev(c["cache_start"]), u32(c["ro"]), dev(base, torch.int64),
                               dev(idx), scale, n_append=n_append, append_base=dev(base, torch.int64) if n_append else None,
                               row_pos_add=n_append, lse=lse, dev_status=status)
    assert status.item() == 0
    ref = omla.sparse_mla(c["q"], lat_deq, c["cache_start"], c["row_req"], idx, scale, n_append=n_append,
                          append_base=base if n_append else None)
    o = out.float().cpu().numpy()
    ls = lse.cpu().numpy()
    worst = 0.0
    for r in range(R):
        worst = max(worst, parity.check_attention_row(o[r], ref[r][0], parity.ATT_TOL_BF16))
        assert np.max(np.abs(ls[r] - ref[r][1])) <= 2e-3 * max(1.0, np.max(np.abs(ref[r][1])))
    print(f"worst relative L2 error {worst:.2e}")


def test_writeback_fp8_latent_rows(mt):
    rng = np.random.default_rng(8)
    B, Wn, T = 20, 6, 2000
    src = rng.integers(0, 256, (B, Wn, 656), dtype=np.uint8)
    dst = rng.integers(0, 256, (T, 656), dtype=np.uint8)
    n_acc = rng.integers(0, Wn, B).astype(np.int32)
    start = (np.arange(B) * 90).astype(np.int64)
    g_dst = dev(dst)
    mt.kv_writeback(dev(src), None, None, dev(n_acc), g_dst, None, None, dev(np.zeros(B, np.int64)), dev(start))
    want = owb.kv_writeback(src, np.zeros((B, Wn, 16), np.uint8), np.zeros((B, Wn), np.float32),
                            np.minimum(n_acc + 1, Wn), dst, np.zeros((T, 16), np.uint8), np.zeros(T, np.float32),
                            start)[0]
    assert g_dst.cpu().numpy().tobytes() == want.tobytes()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_sparse_mla_append_and_edges(mt, dtype):
    """Shared-index draft steps (appended positions), -1 padding, empty rows and
    out-of-range indices (skipped and flagged)."""
    c = _mla_case(64, [500, 60], 128, dtype, seed=7, n_rows=1)
    R = 2
    scale = 1.0 / math.sqrt(576.0)
    idx = c["idx"].copy()
    idx[1, :] = -1                                   # empty selection
    base = c["row_pos"].astype(np.int64)             # step-0 positions; steps append base+1..base+j
    for j in (0, 1, 3):
        lse = torch.empty(R, 64, device="cuda")
        out = mt.sparse_mla_decode(dev(c["q"]), dev(c["latent"]), dev(c["cache_start"]), u32(c["ro"]),
                                   dev(base, torch.int64), dev(idx), scale, n_append=j,
                                   append_base=dev(base, torch.int64) if j else None, row_pos_add=j, lse=lse)
        ref = omla.sparse_mla(c["q"], c["latent"], c["cache_start"], c["row_req"], idx, scale,
                              n_append=j, append_base=base)
        tol = parity.ATT_TOL_F32 if dtype == torch.float32 else parity.ATT_TOL_BF16
        o = out.float().cpu().numpy()
        for r in range(R):
            if j == 0 and r == 1:
                assert np.all(o[r] == 0) and np.all(np.isneginf(lse[r].cpu().numpy()))
            else:
                parity.check_attention_row(o[r], ref[r][0], tol)
    # an index beyond the row position is skipped and flagged
    bad = idx.copy()
    bad[0, 0] = int(base[0]) + 5
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = mt.sparse_mla_decode(dev(c["q"]), dev(c["latent"]), dev(c["cache_start"]), u32(c["ro"]),
                               dev(base, torch.int64), dev(bad), scale, dev_status=status)
    skip = bad.copy()
    skip[0, 0] = -1
    ref = omla.sparse_mla(c["q"], c["latent"], c["cache_start"], c["row_req"], skip, scale, rows=[0])
    parity.check_attention_row(out.float().cpu().numpy()[0], ref[0][0],
                               parity.ATT_TOL_F32 if dtype == torch.float32 else parity.ATT_TOL_BF16)
    assert status.item() & 1
