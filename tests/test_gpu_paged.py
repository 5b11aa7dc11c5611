"""Paged (slotted) KV caches through the C ABI against the oracle: the window's
slot plan, the accepted-KV move, the write-back by slot, and the indexer and
sparse MLA reading through a block table.  The oracle reads every position
through its own slot map (oracle.paged) and computes on the gathered rows."""
import math

import numpy as np
import pytest
import torch

from oracle import fp8 as ofp8
from oracle import indexer as oindexer
from oracle import mla as omla
from oracle import paged as opaged
from oracle import writeback as owb  # noqa: F401  (kept beside the slot write-back for readers)

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


def paged_layout(caps, ps, rng, spare_pages=3, width_extra=1):
    """A block table for requests of the given capacities (positions): each request gets
    ceil(cap / ps) pages drawn from a shuffled pool with a few spare pages; entries past a
    request's pages are -1.  Returns (block_table [B, n] int32, pool pages)."""
    need = [int(math.ceil(c / ps)) for c in caps]
    n_pages = sum(need) + spare_pages
    perm = rng.permutation(n_pages)
    width = max(need) + width_extra
    bt = np.full((len(caps), width), -1, dtype=np.int32)
    o = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[o:o + n]
        o += n
    return bt, n_pages


def scatter_to_pool(logical, bt, ps, pool_rows, rng):
    """Pool [pool_rows, ...] holding logical[b][s] at slot_of(b, s); other slots hold noise."""
    first = logical[0]
    pool = rng.integers(0, 256, (pool_rows,) + first.shape[1:]).astype(first.dtype) if first.dtype == np.uint8 \
        else rng.normal(size=(pool_rows,) + first.shape[1:]).astype(first.dtype)
    for b, rows in enumerate(logical):
        for s in range(len(rows)):
            t = opaged.slot_of(bt, ps, b, s)
            assert t >= 0
            pool[t] = rows[s]
    return pool


def logical_concat(pool, bt, ps, lens):
    """The oracle's view of a paged cache: each request's positions 0..len-1 read through the slot
    map (oracle.paged.gather_positions) and laid end to end, with their starts."""
    parts = [opaged.gather_positions(pool, bt, ps, b, range(int(n))) for b, n in enumerate(lens)]
    start = np.concatenate([[0], np.cumsum([len(p) for p in parts])[:-1]]).astype(np.int64)
    return np.concatenate(parts), start


# ----------------------------------------------------------------------------- slot plan

@pytest.mark.parametrize("ps", [1, 4, 64])
def test_assign_cache_locs(mt, ps):
    rng = np.random.default_rng(ps)
    B, W = 37, 6
    caps = rng.integers(1, 40 * ps, B)
    bt, _ = paged_layout(caps, ps, rng)
    bt[3, 0] = -1                                  # a hole inside a table
    start = np.minimum(caps - 1, rng.integers(0, 40 * ps, B)).astype(np.int64)
    start[5] = bt.shape[1] * ps - 2                # the window runs past the table's width
    start[3] = 0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = mt.assign_cache_locs(dev(bt), ps, dev(start), W, dev_status=status).cpu().numpy()
    want = opaged.assign_cache_locs(bt, ps, start, W)
    assert np.array_equal(got, want)
    assert (want < 0).any() and status.item() & 8, "a window position without a slot must be flagged"


# ----------------------------------------------------------------------------- accepted-KV move

def test_kv_move_accepted(mt):
    rng = np.random.default_rng(11)
    B, W, ps = 40, 6, 4
    caps = rng.integers(W + 1, 300, B)
    bt, n_pages = paged_layout(caps, ps, rng)
    T = n_pages * ps
    start = (caps - W).astype(np.int64)
    loc = opaged.assign_cache_locs(bt, ps, start, W)
    acc_len = rng.integers(0, W + 1, B).astype(np.int32)
    acc_idx = np.tile(np.arange(W, dtype=np.int32), (B, 1))        # chain: the prefix (no move)
    for b in range(0, B, 3):                                        # tree-like: later rows accepted
        cols = np.sort(rng.choice(W, size=W, replace=False))
        shift = rng.integers(0, W)
        acc_idx[b] = np.roll(cols, -shift) if b % 2 else cols[::-1]
        acc_len[b] = rng.integers(1, W + 1)
    acc_idx[1, :3] = [1, 2, 3]                                      # overlapping lists: a shift left
    acc_len[1] = 3
    acc_idx[2, :2] = [1, 0]                                         # a swap
    acc_len[2] = 2
    lat = torch.randn(T, 576).to(torch.bfloat16)
    keys = torch.from_numpy(rng.integers(0, 256, (T, 128), dtype=np.uint8))
    ksc = torch.rand(T)
    g_l, g_k, g_s = dev(lat), dev(keys), dev(ksc)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mt.kv_move_accepted(g_l, g_k, g_s, dev(loc), dev(acc_idx), dev(acc_len - 1), dev_status=status)
    want = opaged.kv_move_accepted([lat.view(torch.int16).numpy(), keys.numpy(), ksc.numpy()], loc, acc_idx, acc_len)
    assert g_l.cpu().view(torch.int16).numpy().tobytes() == want[0].tobytes()
    assert g_k.cpu().numpy().tobytes() == want[1].tobytes()
    assert g_s.cpu().numpy().tobytes() == want[2].tobytes()
    assert status.item() == 0
    # a window column outside [0, W) is skipped and flagged; other rows still move
    bad_idx = acc_idx.copy()
    bad_idx[4, 0] = W + 3
    bad_len = acc_len.copy()
    bad_len[4] = 1
    g_l2 = dev(lat)
    mt.kv_move_accepted(g_l2, None, None, dev(loc), dev(bad_idx), dev(bad_len - 1), dev_status=status)
    ok_len = bad_len.copy()
    ok_len[4] = 0
    want2 = opaged.kv_move_accepted([lat.view(torch.int16).numpy()], loc, bad_idx, ok_len)
    assert g_l2.cpu().view(torch.int16).numpy().tobytes() == want2[0].tobytes()
    assert status.item() & 1


@pytest.mark.parametrize("lat_kind", ["bf16", "fp8"])
def test_kv_writeback_slots(mt, lat_kind):
    rng = np.random.default_rng(12)
    B, W, ps = 33, 6, 64
    caps = rng.integers(W + 1, 2000, B)
    bt, n_pages = paged_layout(caps, ps, rng)
    T = n_pages * ps
    start = (caps - W).astype(np.int64)
    slots = opaged.assign_cache_locs(bt, ps, start, W)
    slots[7, 0] = T + 5                                   # outside the pool: skipped and flagged
    n_acc = rng.integers(0, W, B).astype(np.int32)
    n_acc[0], n_acc[1] = 0, W - 1
    n_acc[7] = 0
    if lat_kind == "bf16":
        src_l = torch.randn(B, W, 576).to(torch.bfloat16)
        dst_l = torch.randn(T, 576).to(torch.bfloat16)
        view = lambda t: t.view(torch.int16).numpy()      # noqa: E731
    else:
        src_l = torch.from_numpy(rng.integers(0, 256, (B, W, 656), dtype=np.uint8))
        dst_l = torch.from_numpy(rng.integers(0, 256, (T, 656), dtype=np.uint8))
        view = lambda t: t.numpy()                        # noqa: E731
    src_k = torch.from_numpy(rng.integers(0, 256, (B, W, 128), dtype=np.uint8))
    src_s = torch.rand(B, W)
    dst_k = torch.from_numpy(rng.integers(0, 256, (T, 128), dtype=np.uint8))
    dst_s = torch.rand(T)
    g_l, g_k, g_s = dev(dst_l), dev(dst_k), dev(dst_s)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int64, device="cuda")
    mt.kv_writeback_slots(dev(src_l), dev(src_k), dev(src_s), dev(n_acc), g_l, g_k, g_s, dev(slots), dev(start),
                          nxt, dev_status=status)
    assert np.array_equal(nxt.cpu().numpy(), start + np.minimum(n_acc + 1, W))
    acc = np.minimum(n_acc + 1, W)
    acc[7] = 0                                            # its only row targets a slot outside the pool
    wl, wk, ws = opaged.kv_writeback_slots(view(src_l), src_k.numpy(), src_s.numpy(), acc, view(dst_l),
                                           dst_k.numpy(), dst_s.numpy(), slots)
    assert view(g_l.cpu()).tobytes() == wl.tobytes()
    assert g_k.cpu().numpy().tobytes() == wk.tobytes()
    assert g_s.cpu().numpy().tobytes() == ws.tobytes()
    assert status.item() & 2


# ----------------------------------------------------------------------------- indexer over a paged cache

@pytest.mark.parametrize("H,D,lens,r_per,k,fp8,ps", [
    (64, 128, [300, 1000, 129, 5], 6, 256, True, 64),     # tensor-core kernel, two boxes per key tile
    (64, 128, [4100, 200], 1, 2048, True, 8),             # 16 boxes of 8 rows per tile
    (64, 128, [3000, 700], 6, 2048, True, 256),           # pages larger than a tile
    (32, 128, [777, 1500, 64], 3, 512, True, 16),
    (64, 128, [500, 300], 2, 128, True, 1),               # the token table itself (CUDA-core kernel)
    (4, 64, [100, 300], 4, 32, False, 4),                 # float32
])
def test_indexer_paged(mt, H, D, lens, r_per, k, fp8, ps):
    rng = np.random.default_rng(H + k + ps)
    B = len(lens)
    caps = np.asarray(lens) + r_per
    bt, n_pages = paged_layout(caps, ps, rng)
    T = n_pages * ps
    row_req = np.repeat(np.arange(B), r_per)
    row_pos = np.repeat(lens, r_per) + np.tile(np.arange(r_per), B)
    R = len(row_req)
    q = rng.normal(size=(R, H, D)).astype(np.float32)
    w = rng.uniform(0, 1, (R, H)).astype(np.float32)
    w[0, 0] = -0.5
    logical = [rng.normal(size=(int(c), D)).astype(np.float32) for c in caps]
    ro = np.concatenate([[0], np.cumsum(np.full(B, r_per))]).astype(np.uint32)
    maxv = int(row_pos.max()) + 1
    if fp8:
        k_pool = scatter_to_pool(logical, bt, ps, T, rng)
        kc, ks = ofp8.quantize_block128(k_pool)
        qc, qs = ofp8.quantize_block128(q)
        qs, ks = qs[..., 0], ks[:, 0]
        gq, gqs, gk, gks = dev(qc), dev(qs), dev(kc), dev(ks)
        lk, lstart = logical_concat(kc, bt, ps, caps)
        lks, _ = logical_concat(ks, bt, ps, caps)
        ref = oindexer.indexer_scores(qc, qs, w, lk, lks, lstart, row_req, row_pos, fp8=True)
    else:
        k_pool = scatter_to_pool(logical, bt, ps, T, rng)
        gq, gqs, gk, gks = dev(q), None, dev(k_pool), None
        lk, lstart = logical_concat(k_pool, bt, ps, caps)
        ref = oindexer.indexer_scores(q, None, w, lk, None, lstart, row_req, row_pos, fp8=False)
    ld = mt.scores_ld(maxv)
    scores = torch.full((R, ld), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = mt.indexer_topk(gq, gqs, dev(w), gk, gks, None, u32(ro), dev(row_pos, torch.int64), k, maxv,
                          scores=scores, dev_status=status, paged=(dev(bt), ps)).cpu().numpy()
    assert status.item() == 0
    sc = scores.cpu().numpy()
    for r in range(R):
        V = int(row_pos[r]) + 1
        parity.check_scores_row(sc[r, :V], ref[r])
        parity.check_topk_row(idx[r], ref[r], k)
    # the contiguous layout of the same keys gives bit-identical scores when the same kernel serves
    # both (FP8 pages under 8 tokens take the CUDA-core kernel, the contiguous call the tensor cores)
    if fp8 and ps < 8:
        return
    if fp8:
        ck, cks = dev(lk), dev(lks)
    else:
        ck, cks = dev(lk), None
    sc2 = mt.indexer_scores(gq, gqs, dev(w), ck, cks, dev(lstart), u32(ro), dev(row_pos, torch.int64), maxv).cpu().numpy()
    for r in range(R):
        V = int(row_pos[r]) + 1
        assert np.array_equal(sc2[r, :V].view(np.uint32), sc[r, :V].view(np.uint32)), f"row {r}"


@pytest.mark.parametrize("ps", [64, 1])
def test_indexer_paged_missing_page(mt, ps):
    """A visible position whose page is missing scores 0 (zero keys) and is flagged."""
    rng = np.random.default_rng(5 + ps)
    H, D, B, r_per = 64, 128, 2, 2
    lens = [700, 400]
    caps = np.asarray(lens) + r_per
    bt, n_pages = paged_layout(caps, ps, rng)
    T = n_pages * ps
    hole = 3 if ps == 64 else 200                     # page index inside request 0's visible range
    bt_hole = bt.copy()
    bt_hole[0, hole] = -1
    row_req = np.repeat(np.arange(B), r_per)
    row_pos = np.repeat(lens, r_per) + np.tile(np.arange(r_per), B)
    R = len(row_req)
    q = rng.normal(size=(R, H, D)).astype(np.float32)
    w = rng.uniform(0, 1, (R, H)).astype(np.float32)
    logical = [rng.normal(size=(int(c), D)).astype(np.float32) for c in caps]
    kc, ks = ofp8.quantize_block128(scatter_to_pool(logical, bt, ps, T, rng))
    qc, qs = ofp8.quantize_block128(q)
    qs, ks = qs[..., 0], ks[:, 0]
    ro = np.concatenate([[0], np.cumsum(np.full(B, r_per))]).astype(np.uint32)
    maxv = int(row_pos.max()) + 1
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc = mt.indexer_scores(dev(qc), dev(qs), dev(w), dev(kc), dev(ks), None, u32(ro), dev(row_pos, torch.int64), maxv,
                           dev_status=status, paged=(dev(bt_hole), ps)).cpu().numpy()
    assert status.item() & 8
    # the oracle over the same table with the missing page's keys and scales read as zeros
    lk, lstart = logical_concat(kc, bt, ps, caps)
    lks, _ = logical_concat(ks, bt, ps, caps)
    gone = np.arange(hole * ps, (hole + 1) * ps)
    lk[gone] = 0
    lks[gone] = 0.0
    ref = oindexer.indexer_scores(qc, qs, w, lk, lks, lstart, row_req, row_pos, fp8=True)
    for r in range(R):
        V = int(row_pos[r]) + 1
        parity.check_scores_row(sc[r, :V], ref[r])
        if row_req[r] == 0:
            assert np.all(sc[r, gone[gone < V]] == 0.0)


# ----------------------------------------------------------------------------- sparse MLA over a paged cache

@pytest.mark.parametrize("H,lens,n_idx,kind,ps,n_append", [
    (128, [300, 2100, 50], 512, "bf16", 64, 0),           # tensor-core kernel
    (128, [9000], 2048, "bf16", 1, 0),                    # token table, several splits
    (128, [5000, 64], 2048, "bf16", 16, 2),               # appended positions (shared draft steps)
    (16, [700, 40], 256, "bf16", 8, 0),                   # mma.sync kernel
    (8, [100, 300], 32, "f32", 4, 0),
    (128, [3000, 64], 1024, "fp8", 32, 1),                # the 656-byte FP8 latent rows
    (128, [2500, 700], 1024, "persist", 64, 0),           # the persistent launch (rows cut between clusters)
    (128, [5000, 64], 2048, "persist", 8, 2),
])
def test_sparse_mla_paged(mt, H, lens, n_idx, kind, ps, n_append, monkeypatch):
    if kind == "persist":
        monkeypatch.setenv("MTPSD_MLA_PERSIST", "1")
    rng = np.random.default_rng(H + n_idx + ps)
    B, n_rows = len(lens), 3
    caps = np.asarray(lens) + n_rows + n_append + 1
    bt, n_pages = paged_layout(caps, ps, rng)
    T = n_pages * ps
    row_req = np.repeat(np.arange(B), n_rows)
    base = np.repeat(lens, n_rows) + np.tile(np.arange(n_rows), B)      # positions of the rows (step 0)
    R = len(row_req)
    g = torch.Generator().manual_seed(H + n_idx)
    tdt = torch.float32 if kind == "f32" else torch.bfloat16
    lat_pool_t = torch.randn(T, 576, generator=g).to(tdt)
    q = torch.randn(R, H, 576, generator=g).to(tdt)
    idx = np.full((R, n_idx), -1, dtype=np.int32)
    for r in range(R):
        V = int(base[r]) + 1
        sel = np.sort(rng.choice(V, size=min(V, n_idx), replace=False))
        idx[r, :len(sel)] = sel
    ro = np.concatenate([[0], np.cumsum(np.full(B, n_rows))]).astype(np.uint32)
    if kind == "fp8":
        lat_g = mt.pack_latent_fp8(dev(lat_pool_t))
        lat_ref_pool = omla.unpack_fp8_ds_mla(omla.pack_fp8_ds_mla(lat_pool_t.float().numpy()))
    else:
        lat_g = dev(lat_pool_t)
        lat_ref_pool = lat_pool_t.float().numpy()
    scale = 1.0 / math.sqrt(576.0)
    lse = torch.empty(R, H, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = mt.sparse_mla_decode(dev(q), lat_g, None, u32(ro), dev(base, torch.int64), dev(idx), scale,
                               n_append=n_append, append_base=dev(base, torch.int64) if n_append else None,
                               row_pos_add=n_append, lse=lse, dev_status=status, paged=(dev(bt), ps))
    assert status.item() == 0
    lat_log, lstart = logical_concat(lat_ref_pool, bt, ps, caps)
    ref = omla.sparse_mla(q, lat_log, lstart, row_req, idx, scale, n_append=n_append,
                          append_base=base if n_append else None)
    tol = parity.ATT_TOL_F32 if kind == "f32" else parity.ATT_TOL_BF16
    o = out.float().cpu().numpy()
    ls = lse.cpu().numpy()
    for r in range(R):
        parity.check_attention_row(o[r], ref[r][0], tol)
        assert np.max(np.abs(ls[r] - ref[r][1])) <= (1e-4 if kind == "f32" else 2e-3) * max(
            1.0, np.max(np.abs(ref[r][1])))


def test_sparse_mla_paged_missing_page(mt):
    """A selected position whose page is missing is skipped and flagged; the rest attends as usual."""
    rng = np.random.default_rng(77)
    H, lens, n_idx, ps = 128, [900, 300], 256, 16
    B = len(lens)
    caps = np.asarray(lens) + 2
    bt, n_pages = paged_layout(caps, ps, rng)
    T = n_pages * ps
    row_req = np.arange(B)
    base = np.asarray(lens, dtype=np.int64)
    g = torch.Generator().manual_seed(3)
    lat = torch.randn(T, 576, generator=g).to(torch.bfloat16)
    q = torch.randn(B, H, 576, generator=g).to(torch.bfloat16)
    idx = np.stack([np.sort(rng.choice(int(base[r]) + 1, n_idx, replace=False)) for r in range(B)]).astype(np.int32)
    page = int(idx[0, 10]) // ps
    bt_hole = bt.copy()
    bt_hole[0, page] = -1
    ro = np.arange(B + 1, dtype=np.uint32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = mt.sparse_mla_decode(dev(q), dev(lat), None, u32(ro), dev(base), dev(idx), 1.0 / math.sqrt(576.0),
                               dev_status=status, paged=(dev(bt_hole), ps))
    assert status.item() & 8
    skip = idx.copy()
    skip[0, idx[0] // ps == page] = -1
    lat_log, lstart = logical_concat(lat.float().numpy(), bt, ps, caps)
    ref = omla.sparse_mla(q, lat_log, lstart, row_req, skip, 1.0 / math.sqrt(576.0))
    o = out.float().cpu().numpy()
    for r in range(B):
        parity.check_attention_row(o[r], ref[r][0], parity.ATT_TOL_BF16)
