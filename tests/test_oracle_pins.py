"""Pins of the CPU oracle against facts fixed outside the oracle itself:
a library codec, hand-worked examples, closed forms, brute force and
textbook dense attention.  CPU only."""
import itertools
import math

import numpy as np
import pytest
import torch

from oracle import accept, fp8, indexer, merge, mla, paged, share, topk, writeback


# --------------------------------------------------------------------- FP8 codec

def test_fp8_decode_exhaustive_vs_library():
    codes = np.arange(256, dtype=np.uint8)
    ours = fp8.decode_e4m3(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan_ours = np.isnan(ours)
    assert np.array_equal(nan_ours, np.isnan(lib))
    assert np.array_equal(ours[~nan_ours], lib[~nan_ours])
    # hand-checked code points of the OCP E4M3 table
    assert fp8.decode_e4m3(np.uint8(0x7E)) == 448.0
    assert fp8.decode_e4m3(np.uint8(0x01)) == 2.0 ** -9
    assert fp8.decode_e4m3(np.uint8(0x08)) == 2.0 ** -6
    assert fp8.decode_e4m3(np.uint8(0x38)) == 1.0
    assert fp8.decode_e4m3(np.uint8(0xB8)) == -1.0
    assert np.isnan(fp8.decode_e4m3(np.uint8(0x7F))) and np.isnan(fp8.decode_e4m3(np.uint8(0xFF)))


def test_fp8_encode_matches_library_rounding():
    rng = np.random.default_rng(0)
    y = np.concatenate([rng.normal(0, 50, 20000), rng.uniform(-448, 448, 20000),
                        rng.normal(0, 0.01, 5000)]).astype(np.float32)
    y = np.concatenate([y, np.array([0.0, -0.0, -1e-6, 1e-6, -0.0009], np.float32)])
    ours = fp8.encode_e4m3_rne_satfinite(y.astype(np.float64))
    lib = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, lib)          # code for code, signed zeros included


def test_fp8_encode_ties_and_saturation():
    # 1.0625 is halfway between 1.0 (0x38, even) and 1.125 (0x39): ties to even
    assert fp8.encode_e4m3_rne_satfinite(np.array([1.0625]))[0] == 0x38
    # 1.1875 is halfway between 1.125 (0x39) and 1.25 (0x3A): ties to even
    assert fp8.encode_e4m3_rne_satfinite(np.array([1.1875]))[0] == 0x3A
    assert fp8.encode_e4m3_rne_satfinite(np.array([1000.0]))[0] == 0x7E
    assert fp8.encode_e4m3_rne_satfinite(np.array([-1000.0]))[0] == 0xFE
    # every finite code round-trips
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    back = fp8.encode_e4m3_rne_satfinite(fp8.decode_e4m3(codes))
    dec = fp8.decode_e4m3(back)
    assert np.array_equal(dec, fp8.decode_e4m3(codes))


def test_quantize_block128_definition():
    rng = np.random.default_rng(1)
    x = rng.normal(0, 3, (5, 256)).astype(np.float32)
    x[2, :128] = 0.0                                   # amax = 0 block
    codes, scale = fp8.quantize_block128(x)
    assert codes.shape == x.shape and scale.shape == (5, 2)
    assert scale[2, 0] == 1.0 and np.all(codes[2, :128] == 0)
    amax = np.abs(x.reshape(5, 2, 128)).max(-1)
    nz = amax > 0
    assert np.array_equal(scale[nz], (amax / np.float32(448.0)).astype(np.float32)[nz])
    # the block maximum maps to +-448 and the library codec agrees per element
    y = (x.reshape(5, 2, 128) / scale[..., None]).astype(np.float32).reshape(5, 256)
    lib = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, lib)
    deq = fp8.decode_e4m3(codes).reshape(5, 2, 128) * scale[..., None]
    assert np.max(np.abs(deq).max(-1)[nz] - amax[nz]) <= 1e-6 * amax.max()


# --------------------------------------------------------------------- merge

def test_merge_hand_worked():
    # two requests with 2 and 1 prompt tokens, K = 3 drafts each
    prompt = np.array([10, 11, 20])
    po = np.array([0, 2, 3], dtype=np.uint32)
    draft = np.array([[1, 2, 3], [4, 5, 6]])
    toks, mo = merge.merge_tokens(prompt, po, draft)
    assert mo.tolist() == [0, 5, 9]
    assert toks.tolist() == [10, 11, 1, 2, 3, 20, 4, 5, 6]
    assert merge.host_merged_offsets(po, 3).tolist() == [0, 5, 9]


def test_merge_k0_identity_and_empty():
    prompt = np.array([7, 8, 9, 10])
    po = np.array([0, 1, 4], dtype=np.uint32)
    toks, mo = merge.merge_tokens(prompt, po, np.zeros((2, 0), dtype=np.int64))
    assert toks.tolist() == [7, 8, 9, 10] and mo.tolist() == [0, 1, 4]
    toks, mo = merge.merge_tokens(np.zeros(0, dtype=np.int64), np.array([0, 0, 0], dtype=np.uint32),
                                  np.array([[1, 2], [3, 4]]))
    assert toks.tolist() == [1, 2, 3, 4] and mo.tolist() == [0, 2, 4]


# --------------------------------------------------------------------- indexer

def test_indexer_hand_worked():
    # H = 2 heads, D = 2.  q = [[1, 2], [-1, 1]], key = [3, 1]:
    # head dots 5 and -2 -> ReLU 5 and 0; w = [0.5, 2] -> 2.5
    q = np.array([[[1.0, 2.0], [-1.0, 1.0]]])
    w = np.array([[0.5, 2.0]])
    k = np.array([[3.0, 1.0], [-1.0, 0.0], [0.0, 0.0]])
    out = indexer.indexer_scores(q, None, w, k, None, np.array([0]), np.array([0]),
                                 np.array([2]), fp8=False)
    # key 1: dots -1 and 1 -> 0 + 2*1 = 2; key 2: all zero -> 0
    assert out[0].tolist() == [2.5, 2.0, 0.0]


def test_indexer_brute_force_loops_and_visibility():
    rng = np.random.default_rng(2)
    H, D, T = 3, 8, 40
    q = rng.normal(size=(4, H, D))
    w = rng.uniform(-1, 1, size=(4, H))      # negative weights stay outside the ReLU
    k = rng.normal(size=(T, D))
    cache_start = np.array([0, 17])
    row_req = np.array([0, 0, 1, 1])
    row_pos = np.array([10, 11, 20, 22])
    out = indexer.indexer_scores(q, None, w, k, None, cache_start, row_req, row_pos, fp8=False)
    for r in range(4):
        base = cache_start[row_req[r]]
        assert len(out[r]) == row_pos[r] + 1
        for s in range(row_pos[r] + 1):
            tot = 0.0
            for h in range(H):
                d = sum(q[r, h, i] * k[base + s, i] for i in range(D))
                if d > 0:
                    tot += w[r, h] * d
            assert abs(out[r][s] - tot) <= 1e-12 * max(1.0, abs(tot))


def test_indexer_fp8_scales_commute_with_relu():
    rng = np.random.default_rng(3)
    H, D, T = 4, 128, 50
    qx = rng.normal(size=(1, H, D)).astype(np.float32)
    kx = rng.normal(size=(T, D)).astype(np.float32)
    w = rng.uniform(0, 1, size=(1, H)).astype(np.float32)
    qc, qs = fp8.quantize_block128(qx)
    kc, ks = fp8.quantize_block128(kx)
    ks = ks[:, 0]
    qs = qs[..., 0]
    out = indexer.indexer_scores(qc, qs, w, kc, ks, np.array([0]), np.array([0]),
                                 np.array([T - 1]), fp8=True)[0]
    # same thing with the scales folded outside the ReLU (positive scales commute)
    dots = fp8.decode_e4m3(kc) @ fp8.decode_e4m3(qc[0]).T            # [T, H]
    alt = ks.astype(np.float64) * (np.maximum(dots, 0) @ (w[0].astype(np.float64) * qs[0]))
    assert np.allclose(out, alt, rtol=1e-12, atol=0)
    # and it approximates the unquantized score to FP8 accuracy
    exact = np.maximum(kx.astype(np.float64) @ qx[0].T.astype(np.float64), 0) @ w[0]
    assert np.max(np.abs(out - exact)) < 0.1 * np.max(np.abs(exact))


def test_indexer_single_head_is_plain_dot():
    rng = np.random.default_rng(4)
    k = np.abs(rng.normal(size=(9, 5)))
    q = np.abs(rng.normal(size=(1, 1, 5)))
    out = indexer.indexer_scores(q, None, np.ones((1, 1)), k, None, np.array([0]),
                                 np.array([0]), np.array([8]), fp8=False)[0]
    assert np.allclose(out, np.dot(k, q[0, 0]), rtol=1e-14)


# --------------------------------------------------------------------- top-k

def _brute_topk(scores, k):
    """Best subset by exhaustive search: the k-subset with the largest sorted
    score vector, ties to the subset with smaller positions."""
    V = len(scores)
    best = None
    for sub in itertools.combinations(range(V), min(k, V)):
        key = (sorted((scores[i] for i in sub), reverse=True), [-i for i in sorted(sub)])
        if best is None or key > best[0]:
            best = (key, sub)
    return sorted(best[1])


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(5)
    for trial in range(40):
        V = int(rng.integers(1, 10))
        k = int(rng.integers(1, 8))
        scores = rng.integers(0, 4, V).astype(np.float64)     # many exact ties
        got = topk.topk_select(scores, k)
        want = _brute_topk(scores, k)
        assert got[:len(want)].tolist() == want
        assert np.all(got[len(want):] == -1)


def test_topk_short_row_takes_all():
    got = topk.topk_select(np.array([0.5, -1.0, 2.0]), 8)
    assert got.tolist() == [0, 1, 2, -1, -1, -1, -1, -1]


def test_topk_ties_to_lower_index():
    got = topk.topk_select(np.array([1.0, 3.0, 1.0, 1.0, 0.0]), 3)
    assert got.tolist() == [0, 1, 2]


# --------------------------------------------------------------------- sparse MLA

def _dense_attention(q, C, scale):
    """Textbook softmax attention with torch in float64: q [H, 576], C [n, 576]."""
    qt = torch.from_numpy(np.asarray(q, dtype=np.float64))
    Ct = torch.from_numpy(np.asarray(C, dtype=np.float64))
    logits = scale * qt @ Ct.T
    p = torch.softmax(logits, dim=-1)
    return (p @ Ct[:, :512]).numpy(), torch.logsumexp(logits, dim=-1).numpy()


def test_sparse_mla_equals_dense_when_k_covers_context():
    rng = np.random.default_rng(6)
    H, T = 4, 60
    latent = rng.normal(size=(T, 576))
    q = rng.normal(size=(3, H, 576))
    cache_start = np.array([0, 25])
    row_req = np.array([0, 1, 1])
    row_pos = np.array([20, 30, 34])
    k = 64
    idx = np.full((3, k), -1)
    for r in range(3):
        idx[r, :row_pos[r] + 1] = rng.permutation(row_pos[r] + 1)   # any order
    out = mla.sparse_mla(q, latent, cache_start, row_req, idx, 0.07)
    for r in range(3):
        base = cache_start[row_req[r]]
        o_ref, lse_ref = _dense_attention(q[r], latent[base:base + row_pos[r] + 1], 0.07)
        assert np.allclose(out[r][0], o_ref, rtol=1e-12, atol=1e-13)
        assert np.allclose(out[r][1], lse_ref, rtol=1e-12)


def test_sparse_mla_closed_forms():
    rng = np.random.default_rng(7)
    latent = rng.normal(size=(20, 576))
    q = rng.normal(size=(1, 2, 576))
    # one selected row: output is that row's first 512 values, lse = its logit
    idx = np.array([[7, -1, -1]])
    o, lse = mla.sparse_mla(q, latent, np.array([0]), np.array([0]), idx, 0.1)[0]
    assert np.allclose(o, latent[7, :512][None].repeat(2, 0), rtol=1e-14)
    assert np.allclose(lse, 0.1 * latent[7] @ q[0].T, rtol=1e-13)
    # q = 0: uniform weights, the mean of the selected rows; lse = log n
    idx = np.array([[3, 9, 11, 4]])
    o, lse = mla.sparse_mla(np.zeros((1, 1, 576)), latent, np.array([0]), np.array([0]), idx, 1.0)[0]
    assert np.allclose(o[0], latent[[3, 9, 11, 4], :512].mean(0), rtol=1e-13)
    assert np.allclose(lse, math.log(4.0))
    # empty selection
    o, lse = mla.sparse_mla(q, latent, np.array([0]), np.array([0]), np.full((1, 4), -1), 0.1)[0]
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_sparse_mla_appended_positions():
    rng = np.random.default_rng(8)
    latent = rng.normal(size=(30, 576))
    q = rng.normal(size=(1, 2, 576))
    idx = np.array([[2, 5, -1]])
    got = mla.sparse_mla(q, latent, np.array([3]), np.array([0]), idx, 0.05,
                         n_append=2, append_base=np.array([10]))[0]
    want = mla.sparse_mla(q, latent, np.array([3]), np.array([0]),
                          np.array([[2, 5, 11, 12]]), 0.05)[0]
    assert np.allclose(got[0], want[0], rtol=1e-14) and np.allclose(got[1], want[1], rtol=1e-14)


# --------------------------------------------------------------------- acceptance

def test_accept_hand_worked():
    draft = np.array([[5, 6, 7], [5, 6, 7], [5, 6, 7], [42, 42, 42], [1, 2, 3]])
    tgt = np.array([[5, 6, 7, 99],      # all match -> 3, bonus 99
                    [9, 6, 7, 99],      # mismatch at 0 -> 0, next 9
                    [5, 6, 8, 99],      # mismatch at 2 -> 2, next 8
                    [42, 42, 42, 77],   # sentinel row -> 0 accepted, next = argmax[0]
                    [1, 2, 3, 4]])
    n, nxt = accept.accept_greedy(draft, tgt, magic_draft_id=42)
    assert n.tolist() == [3, 0, 2, 0, 3]
    assert nxt.tolist() == [99, 9, 8, 42, 4]
    n, nxt = accept.accept_greedy(draft, tgt, magic_draft_id=-1)
    assert n.tolist() == [3, 0, 2, 3, 3]


def test_accept_k0():
    n, nxt = accept.accept_greedy(np.zeros((2, 0), dtype=np.int64), np.array([[3], [4]]))
    assert n.tolist() == [0, 0] and nxt.tolist() == [3, 4]


def test_accept_length_closed_form():
    # synthetic acceptance with per-position probability p: mean accept length
    # 1 + sum_{i=1..K} p^i = 2.76 for p = 0.67065, K = 5
    from mtp_speculative_decode_gb300 import workloads as W
    p, K = W.ACCEPT_P, 5
    assert abs(1 + sum(p ** i for i in range(1, K + 1)) - 2.76) < 1e-3
    import torch as _t
    B = 200000
    draft = W.integers(11, "draft_tokens", (B, K), 0, W.GLM_VOCAB)
    tgt = W.synthetic_argmax(11, draft, W.GLM_VOCAB, p).numpy()
    d = draft.numpy()
    match = d == tgt[:, :K]
    n = np.argmin(np.concatenate([match, np.zeros((B, 1), bool)], 1), axis=1)
    mean = 1 + n.mean()
    assert abs(mean - 2.76) < 4 * n.std() / math.sqrt(B) + 1e-3
    # the oracle agrees with this direct count on a slice
    n2, _ = accept.accept_greedy(d[:500], tgt[:500])
    assert np.array_equal(n2, n[:500])


# --------------------------------------------------------------------- write-back

def test_writeback_bytes():
    rng = np.random.default_rng(9)
    B, W, T = 3, 6, 40
    src_l = rng.normal(size=(B, W, 576)).astype(np.float32)
    src_k = rng.integers(0, 256, (B, W, 128), dtype=np.uint8)
    src_s = rng.uniform(size=(B, W)).astype(np.float32)
    dst_l = rng.normal(size=(T, 576)).astype(np.float32)
    dst_k = rng.integers(0, 256, (T, 128), dtype=np.uint8)
    dst_s = rng.uniform(size=T).astype(np.float32)
    acc = np.array([1, 6, 3])
    start = np.array([2, 10, 30])
    ol, ok, os_ = writeback.kv_writeback(src_l, src_k, src_s, acc, dst_l, dst_k, dst_s, start)
    written = np.zeros(T, bool)
    for b in range(B):
        for i in range(acc[b]):
            t = start[b] + i
            written[t] = True
            assert ol[t].tobytes() == src_l[b, i].tobytes()
            assert ok[t].tobytes() == src_k[b, i].tobytes()
            assert os_[t].tobytes() == src_s[b, i].tobytes()
    assert ol[~written].tobytes() == dst_l[~written].tobytes()
    assert ok[~written].tobytes() == dst_k[~written].tobytes()
    assert os_[~written].tobytes() == dst_s[~written].tobytes()
    assert written.sum() == 1 + 6 + 3


# --------------------------------------------------------------------- index sharing

def test_share_gather_rows():
    s0 = np.arange(12).reshape(6, 2)
    ro = np.array([0, 2, 6])
    assert share.topk_share_gather(s0, ro, np.array([1, 3])).tolist() == [[2, 3], [10, 11]]
    assert share.topk_share_gather(s0, ro, None).tolist() == [[0, 1], [4, 5]]


def test_shared_steps_equal_rerun_when_context_below_k():
    """When P_b + j + 1 <= k the indexer selects everything visible, so the
    shared set plus the appended positions equals rerunning the indexer."""
    rng = np.random.default_rng(10)
    H, D, P = 2, 16, 30
    k_cache = rng.normal(size=(P + 8, D))
    k = 64
    q0 = rng.normal(size=(1, H, D))
    s0 = topk.topk_select(indexer.indexer_scores(q0, None, np.ones((1, H)), k_cache, None,
                                                 np.array([0]), np.array([0]), np.array([P]),
                                                 fp8=False)[0], k)
    for j in range(1, 4):
        qj = rng.normal(size=(1, H, D))
        rerun = topk.topk_select(indexer.indexer_scores(qj, None, np.ones((1, H)), k_cache, None,
                                                        np.array([0]), np.array([0]),
                                                        np.array([P + j]), fp8=False)[0], k)
        shared = share.shared_step_positions(s0, P, j)
        assert sorted(shared) == sorted(int(x) for x in rerun if x >= 0)


# --------------------------------------------------------------------- k-th score (tie band)

def test_kth_score_hand_worked():
    s = np.array([3.0, 1.0, 4.0, 1.0, 5.0, 9.0, 2.0, 6.0])
    # descending: 9 6 5 4 3 2 1 1
    assert topk.kth_score(s, 1) == 9.0
    assert topk.kth_score(s, 3) == 5.0
    assert topk.kth_score(s, 8) == 1.0
    assert topk.kth_score(s, 20) == 1.0            # fewer than k: the smallest
    t = np.array([2.0, 2.0, 2.0, 1.0])
    assert topk.kth_score(t, 2) == 2.0             # ties count once per position
    assert topk.kth_score(t, 3) == 2.0
    assert topk.kth_score(t, 4) == 1.0
    assert topk.kth_score(np.array([-0.5]), 2048) == -0.5


def test_kth_score_is_the_score_of_the_last_selected():
    """The k-th score equals the smallest score topk_select takes (brute
    force over small rows with ties)."""
    rng = np.random.default_rng(21)
    for _ in range(50):
        V = int(rng.integers(1, 9))
        k = int(rng.integers(1, 10))
        sc = rng.integers(-3, 4, V).astype(np.float64)
        sub = _brute_topk(sc, k)
        assert topk.kth_score(sc, k) == min(sc[i] for i in sub)


# --------------------------------------------------------------------- draft inputs after the write-back

def _marker_step(fp8_keys: bool):
    """Two requests, contexts L = [5, 7], window W = 4 (K = 3).  Pool row t of
    the draft layer holds the constant 100 + t in every element; window row i
    of request b holds -(1 + 10 b + i).  Positions are pool rows minus
    cache_start = [0, 20]."""
    import types

    import torch
    from oracle.pipeline import OracleStep
    T, D = 40, 128
    spec = types.SimpleNamespace(K=3, topk=8, latent_f32=not fp8_keys)
    w = types.SimpleNamespace(spec=spec, L=np.array([5, 7]), cache_start=np.array([0, 20]), tensors={})
    pool_k = np.repeat((100.0 + np.arange(T))[:, None], D, axis=1).astype(np.float32)
    pool_l = np.repeat((100.0 + np.arange(T))[:, None], 576, axis=1).astype(np.float32)
    win = -(1.0 + 10.0 * np.arange(2)[:, None] + np.arange(4)[None, :])          # [B, W]
    d = {"d_k_idx": torch.from_numpy(pool_k),
         "src_k_idx": torch.from_numpy(np.repeat(win[:, :, None], D, axis=2).astype(np.float32)),
         "d_latent": torch.from_numpy(pool_l),
         "src_latent": torch.from_numpy(np.repeat(win[:, :, None], 576, axis=2).astype(np.float32))}
    return OracleStep(w, d)


def test_next_pos_hand_worked():
    """The draft step-0 row sits right after the written-back accepted segment
    (bonus included): P = L + num_accepted + 1."""
    o = _marker_step(False)
    assert o.next_pos(np.array([0, 3])).tolist() == [6, 11]
    assert o.next_pos(np.array([2, 0])).tolist() == [8, 8]


def test_draft_keys_overlay_hand_worked():
    o = _marker_step(False)
    n_acc = np.array([0, 3])
    k0 = o.draft_keys(n_acc, 0, 8)[:, 0]
    # request 0: one accepted row (the bonus) overwrites position 5 only
    assert k0.tolist() == [100, 101, 102, 103, 104, -1, 106, 107]
    k1 = o.draft_keys(n_acc, 1, 12)[:, 0]
    # request 1: positions 7..10 take window rows 0..3; position 11 (= L + n) keeps the pool row
    assert k1.tolist() == [120, 121, 122, 123, 124, 125, 126, -11, -12, -13, -14, 131]
    # a visible prefix that ends inside the segment takes only the rows inside it
    assert o.draft_keys(n_acc, 1, 9)[:, 0].tolist() == [120, 121, 122, 123, 124, 125, 126, -11, -12]


def test_draft_keys_requantized_per_token():
    """With FP8 keys every overlaid row carries its own block-128 scale: a
    constant row c quantizes to the code of +-448 with scale |c|/448 and so
    decodes back to c (to float32 rounding of the scale)."""
    o = _marker_step(True)
    k1 = o.draft_keys(np.array([0, 3]), 1, 12)
    want = [120, 121, 122, 123, 124, 125, 126, -11, -12, -13, -14, 131]
    for row, c in zip(k1, want):
        assert np.allclose(row, c, rtol=2 ** -23, atol=0)


def test_draft_latent_rows_overlay_hand_worked():
    o = _marker_step(False)
    n_acc = np.array([1, 0])
    # request 0: accept length 2 -> positions 5, 6 take window rows 0, 1; 7 keeps the pool row
    rows = o.draft_latent_rows(n_acc, 0, [0, 4, 5, 6, 7])
    assert rows[:, 0].tolist() == [100, 104, -1, -2, 107]
    assert rows.shape == (5, 576) and np.all(rows == rows[:, :1])
    # request 1: accept length 1 -> only position 7; position 8 is the pool row (pool row 28)
    rows = o.draft_latent_rows(n_acc, 1, [8, 7, 3])
    assert rows[:, 0].tolist() == [128, -11, 123]


# --------------------------------------------------------------------- stochastic acceptance

def test_accept_stochastic_hand_worked():
    # row 0: p/q = 0.6/0.25 = 2.4 for draft 1, accepted for every u; row 1: p/q = 0.1/0.7 for draft 1
    p = np.array([[[0.1, 0.6, 0.2, 0.1], [0.5, 0.1, 0.2, 0.2], [0.0, 0.0, 0.3, 0.7]]], np.float32)
    q = np.array([[[0.25, 0.25, 0.25, 0.25], [0.1, 0.7, 0.1, 0.1]]], np.float32)
    d = np.array([[1, 1]])
    # u = 0.5 rejects row 1 (0.5 * 0.7 >= 0.1); residual max(0, p1 - q1) = [0.4, 0, 0.1, 0.1], mass 0.6
    n, t = accept.accept_stochastic(d, q, p, np.array([[0.9, 0.5]], np.float32), np.array([0.7], np.float32))
    assert n.tolist() == [1] and t.tolist() == [2]      # 0.7 * 0.6 = 0.42: cumsum 0.4, 0.4, 0.5 -> token 2
    n, t = accept.accept_stochastic(d, q, p, np.array([[0.9, 0.5]], np.float32), np.array([0.5], np.float32))
    assert n.tolist() == [1] and t.tolist() == [0]      # 0.3 < 0.4 -> token 0
    # u = 0.1 accepts row 1 too (0.1 * 0.7 = 0.07 < 0.1): the next token comes from p2 = [0, 0, 0.3, 0.7]
    n, t = accept.accept_stochastic(d, q, p, np.array([[0.0, 0.1]], np.float32), np.array([0.5], np.float32))
    assert n.tolist() == [2] and t.tolist() == [3]      # 0.5 * 1.0 = 0.5: cumsum 0, 0, 0.3, 1.0 -> token 3
    # a draft outside the vocabulary is rejected; an identical draft and target distribution always accepts
    n, t = accept.accept_stochastic(np.array([[9, 1]]), q, p, np.array([[0.0, 0.0]], np.float32),
                                    np.array([0.0], np.float32))
    # residual of row 0 is max(0, p0 - q0) = [0, 0.35, 0, 0]: all its mass is on token 1
    assert n.tolist() == [0] and t.tolist() == [1]
    # p == q accepts whatever u is (u q < q for u < 1)
    n, _ = accept.accept_stochastic(d, p[:, :2], p, np.array([[0.999, 0.999]], np.float32),
                                    np.array([0.3], np.float32))
    assert n.tolist() == [2]


def _spec_sampling_trials(p, q, n_trials, seed):
    """Emitted tokens of n_trials independent one-draft chains (K = 1): the draft
    is drawn from q by inverse CDF, then the oracle decides."""
    rng = np.random.default_rng(seed)
    V = p.shape[-1]
    cq = np.cumsum(q[0].astype(np.float64))
    first, second = [], []
    for _ in range(n_trials):
        d = int(np.searchsorted(cq, rng.random() * cq[-1], side="right"))
        d = min(d, V - 1)
        n, t = accept.accept_stochastic(np.array([[d]]), q[None], p[None],
                                        rng.random((1, 1)).astype(np.float32),
                                        rng.random(1).astype(np.float32))
        if n[0] == 1:
            first.append(d)
            second.append(int(t[0]))
        else:
            first.append(int(t[0]))
    return np.array(first), np.array(second)


def test_accept_stochastic_emits_the_target_distribution():
    """The defining property of speculative sampling (no assumption on how the
    kernel computes it): the first emitted token, accepted draft or corrected
    draw, is distributed exactly as the target p0, whatever q0 is; and after an
    accepted draft the bonus token is distributed as p1."""
    rng = np.random.default_rng(31)
    V = 6
    p = rng.dirichlet(np.ones(V), size=2).astype(np.float32)        # rows 0 and 1 of the target
    q = rng.dirichlet(np.ones(V) * 0.7, size=1).astype(np.float32)  # the draft's row 0
    N = 60000
    first, second = _spec_sampling_trials(p, q, N, 7)
    f1 = np.bincount(first, minlength=V) / N
    sd = np.sqrt(p[0] * (1 - p[0]) / N)
    assert np.all(np.abs(f1 - p[0]) < 5 * sd + 1e-4), (f1, p[0])
    f2 = np.bincount(second, minlength=V) / max(len(second), 1)
    sd2 = np.sqrt(p[1] * (1 - p[1]) / max(len(second), 1))
    assert np.all(np.abs(f2 - p[1]) < 5 * sd2 + 1e-4), (f2, p[1])
    # and the acceptance rate is sum_v min(p0, q0)
    acc_rate = len(second) / N
    want = float(np.minimum(p[0], q[0]).sum())
    assert abs(acc_rate - want) < 5 * np.sqrt(want * (1 - want) / N)


def test_accept_stochastic_inverse_cdf_boundaries():
    w = np.array([0.0, 0.25, 0.0, 0.5, 0.25], np.float32)
    # u * 1.0 against cumulative 0, .25, .25, .75, 1.0: strictly-greater rule
    for u, want in [(0.0, 1), (0.2499, 1), (0.25, 3), (0.7499, 3), (0.75, 4), (0.9999, 4)]:
        assert accept._sample_index(w, u) == want, (u, want)
    assert accept._sample_index(np.zeros(4, np.float32), 0.5) == -1


def test_accept_stochastic_fixed_point_is_exact():
    """The threshold floor(u * total) and the weights floor(w * 2^32) equal the
    exact rational values (fractions.Fraction of the single-precision inputs)."""
    from fractions import Fraction
    rng = np.random.default_rng(5)
    us = np.concatenate([rng.random(200).astype(np.float32),
                         np.array([0.0, 1e-30, 0.5, 0.99999994, 2.0 ** -24, 0.75], np.float32)])
    totals = [1, 3, 2 ** 32, 2 ** 40 + 12345, 154880 * (2 ** 32 - 1), 2 ** 63 - 1]
    for u in us:
        for tot in totals:
            want = int(Fraction(float(u)) * tot)   # floor, both non-negative
            assert accept._scaled_floor(u, tot) == want, (u, tot)
    ws = np.concatenate([rng.random(200).astype(np.float32), np.array([0.0, 1.0, 2.0 ** -40, 3e-10], np.float32)])
    got = accept._fixed_weights(ws)
    assert got == [int(Fraction(float(w)) * 2 ** 32) for w in ws]


# --------------------------------------------------------------------- cross-layer sharing

def test_indexer_schedule_reproduces_the_pages_counts():
    """GLM-5.3's verify step runs the indexer in 21 full layers of 78 and shares it in
    57 ([P2] "验证段的逐层算子"); the automatic rule with frequency 4 and offset 2 gives
    exactly that, with layers 0 and 1 full, then every fourth."""
    t = share.resolve_indexer_types(78, freq=4, offset=2)
    assert t.count("full") == 21 and t.count("shared") == 57
    full = [i for i, x in enumerate(t) if x == "full"]
    assert full[:4] == [0, 1, 5, 9] and full[-1] == 77


def test_indexer_schedule_sources_and_rules():
    assert share.resolve_indexer_types(3) == ["full"] * 3                      # no information
    assert share.resolve_indexer_types(4, pattern="FSSF") == ["full", "shared", "shared", "full"]
    assert share.resolve_indexer_types(2, explicit=["full", "shared"], pattern="FF") == ["full", "shared"]
    assert share.resolve_indexer_types(5, freq=1) == ["full"] * 5              # every layer with frequency 1
    assert share.resolve_indexer_types(6, freq=2, offset=1) == ["full", "shared", "full", "shared", "full", "shared"]
    with pytest.raises(ValueError):
        share.resolve_indexer_types(3, pattern="SFF")                          # first must be full
    with pytest.raises(ValueError):
        share.resolve_indexer_types(3, pattern="FX")
    assert share.source_layers(["full", "shared", "shared", "full", "shared"]) == [0, 0, 0, 3, 3]


def test_seeded_step_positions():
    assert share.seeded_step_positions(np.array([3, 1, -1, 7]), 12) == [3, 1, 7, 12]


def test_seeded_steps_equal_rerun_when_context_below_k():
    """With a context shorter than k the seed (the selection at P - 1) holds every
    position up to P - 1, so the seeded step at P attends exactly what rerunning
    the indexer at P would select: every position 0..P."""
    rng = np.random.default_rng(12)
    H, D, P, k = 2, 16, 40, 64
    keys = rng.normal(size=(P + 4, D))
    seed = topk.topk_select(indexer.indexer_scores(rng.normal(size=(1, H, D)), None, np.ones((1, H)), keys, None,
                                                   np.array([0]), np.array([0]), np.array([P - 1]),
                                                   fp8=False)[0], k)
    rerun = topk.topk_select(indexer.indexer_scores(rng.normal(size=(1, H, D)), None, np.ones((1, H)), keys, None,
                                                    np.array([0]), np.array([0]), np.array([P]), fp8=False)[0], k)
    assert sorted(share.seeded_step_positions(seed, P)) == sorted(int(x) for x in rerun if x >= 0)


# --------------------------------------------------------------------- FP8 latent cache (656 B per token)

def test_fp8_ds_mla_hand_worked_token():
    """One token by hand: latent values 0..511 are block constants c_k (so each
    block's codes are all 448 with scale |c_k|/448, i.e. code 0x7E or 0xFE), the
    rope values are exact bf16 numbers."""
    c = [1.0, -2.5, 448.0, 0.0]
    x = np.zeros((1, 576), np.float32)
    for k in range(4):
        x[0, 128 * k:128 * (k + 1)] = c[k]
    x[0, 512:] = np.arange(64, dtype=np.float32) * 0.5 - 7.0
    pk = mla.pack_fp8_ds_mla(x)
    assert pk.shape == (1, 656) and mla.FP8_DS_MLA_BYTES == 512 + 16 + 128 == 656
    assert set(pk[0, 0:128].tolist()) == {0x7E} and set(pk[0, 128:256].tolist()) == {0xFE}
    assert set(pk[0, 256:384].tolist()) == {0x7E} and set(pk[0, 384:512].tolist()) == {0x00}
    assert pk[0, 512:528].view(np.float32).tolist() == [np.float32(1.0 / 448), np.float32(2.5 / 448), 1.0, 1.0]
    un = mla.unpack_fp8_ds_mla(pk)[0]
    assert np.allclose(un[:512], np.repeat(c, 128), rtol=2 ** -22, atol=0)   # 448 * (c/448) rounded once
    assert np.array_equal(un[512:], x[0, 512:].astype(np.float64))


def test_fp8_ds_mla_round_trip_and_rope_rounding():
    rng = np.random.default_rng(13)
    x = rng.normal(size=(200, 576)).astype(np.float32)
    un = mla.unpack_fp8_ds_mla(mla.pack_fp8_ds_mla(x))
    # E4M3 keeps 3 mantissa bits: |error| <= 2^-4 |x| for normal codes, plus half the smallest
    # subnormal step of the block (2^-10 * scale)
    blk = np.abs(x[:, :512]).reshape(200, 4, 128).max(axis=2) / 448.0
    bound = 2.0 ** -4 * np.abs(x[:, :512]) + 2.0 ** -10 * np.repeat(blk, 128, axis=1) + 1e-30
    assert np.all(np.abs(un[:, :512] - x[:, :512]) <= bound)
    # rope: bf16 of each value, against torch's round-to-nearest-even cast
    import torch
    want = torch.from_numpy(x[:, 512:]).to(torch.bfloat16).double().numpy()
    assert np.array_equal(un[:, 512:], want)


# --------------------------------------------------------------------- the composed step against dense attention

def _composed_step():
    """A hand-built two-request step with k above every context, so that each
    top-k takes every visible position and each attention of the composed
    oracle step must equal textbook dense attention over the rows the readings
    name: contexts L = [6, 9], K = 2 (window W = 3), float32 inputs, and the
    draft-layer pool with the accepted window rows overlaid at L .. L + n - 1."""
    import types

    from oracle.pipeline import OracleStep
    rng = np.random.default_rng(31)
    B, K, W, H_I, D_I, H_Q = 2, 2, 3, 2, 8, 2
    L = np.array([6, 9])
    cap = L + W + 6
    cache_start = np.concatenate([[0], np.cumsum(cap)[:-1]])
    T = int(cap.sum())
    R = B * W
    spec = types.SimpleNamespace(K=K, topk=64, latent_f32=True, draft_steps=3)
    row_req = np.repeat(np.arange(B), W)
    row_pos = np.repeat(L, W) + np.tile(np.arange(W), B)
    f = lambda *s: torch.from_numpy(rng.normal(size=s).astype(np.float32))
    u = lambda *s: torch.from_numpy(rng.uniform(0.1, 1.0, size=s).astype(np.float32))
    t = {"q_idx": f(R, H_I, D_I), "w_idx": u(R, H_I), "k_idx": f(T, D_I), "latent": f(T, 576),
         "q_mla": f(R, H_Q, 576)}
    for l in (1, 2):
        for n, v in (("q_idx", f(R, H_I, D_I)), ("w_idx", u(R, H_I)), ("k_idx", f(T, D_I)), ("latent", f(T, 576)),
                     ("q_mla", f(R, H_Q, 576))):
            t[f"{n}@{l}"] = v
    d = {"d_k_idx": f(T, D_I), "d_latent": f(T, 576), "src_k_idx": f(B, W, D_I), "src_latent": f(B, W, 576),
         "d_q_idx": f(B, H_I, D_I), "d_w_idx": u(B, H_I), "x_q_idx": f(R, H_I, D_I), "x_w_idx": u(R, H_I),
         "x_q_mla": f(R, H_Q, 576)}
    for j in range(spec.draft_steps):
        d[f"d_q_mla{j}"] = f(B, H_Q, 576)
    w = types.SimpleNamespace(spec=spec, L=L, cache_start=cache_start, row_req=row_req, row_pos=row_pos, tensors=t)
    return OracleStep(w, d), w, t, d


def _draft_rows_after_writeback(w, d, b, n_acc, upto):
    """Draft latent rows 0..upto-1 of request b, the first n_acc + 1 window rows written at L_b."""
    base = int(w.cache_start[b])
    rows = d["d_latent"][base:base + upto].double().numpy().copy()
    for i in range(n_acc + 1):
        if w.L[b] + i < upto:
            rows[w.L[b] + i] = d["src_latent"][b, i].double().numpy()
    return rows


def test_composed_verify_and_layers_equal_dense_attention():
    o, w, t, _ = _composed_step()
    scale = 1.0 / math.sqrt(576.0)
    rows = list(range(len(w.row_pos)))
    out = o.verify_mla(o.verify_topk(o.verify_scores(rows)))
    for r in rows:
        base = int(w.cache_start[w.row_req[r]])
        ref = _dense_attention(t["q_mla"][r].double().numpy(),
                               t["latent"][base:base + w.row_pos[r] + 1].double().numpy(), scale)
        assert np.allclose(out[r][0], ref[0], rtol=1e-10, atol=1e-12) and np.allclose(out[r][1], ref[1], rtol=1e-12)
    # full, shared, full: every layer attends its own latent rows 0..p
    _, lo = o.layered_verify(["full", "shared", "full"], rows)
    for l in range(3):
        lat = t["latent"] if l == 0 else t[f"latent@{l}"]
        qm = t["q_mla"] if l == 0 else t[f"q_mla@{l}"]
        for r in rows:
            base = int(w.cache_start[w.row_req[r]])
            ref = _dense_attention(qm[r].double().numpy(), lat[base:base + w.row_pos[r] + 1].double().numpy(), scale)
            assert np.allclose(lo[l][r][0], ref[0], rtol=1e-10, atol=1e-12)


def test_composed_draft_loop_extend_and_seed_equal_dense_attention():
    """Draft step j at P + j = L + n_acc + 1 + j attends rows 0..P+j; draft_extend's
    window row i attends rows 0..L+i; the seeded step j of the next round (seed =
    draft_extend's selection at window row n_acc, position P - 1) attends rows
    0..P+j too: all over the written-back draft pool."""
    o, w, _, d = _composed_step()
    scale = 1.0 / math.sqrt(576.0)
    n_acc = np.array([1, 0])
    P = [int(w.L[b]) + int(n_acc[b]) + 1 for b in range(2)]
    _, shared = o.draft_step0(n_acc, [0, 1])
    _, sel, xo = o.draft_extend(n_acc, [0, 1])
    seed = {b: sel[(b, int(n_acc[b]))] for b in range(2)}
    for j in range(3):
        dm = o.draft_mla(n_acc, shared, j, [0, 1])
        sm = o.seeded_draft_mla(n_acc, seed, j, [0, 1])
        for b in range(2):
            rows = _draft_rows_after_writeback(w, d, b, int(n_acc[b]), P[b] + j + 1)
            ref = _dense_attention(d[f"d_q_mla{j}"][b].double().numpy(), rows, scale)
            assert np.allclose(dm[b][0], ref[0], rtol=1e-10, atol=1e-12), (j, b)
            assert np.allclose(sm[b][0], ref[0], rtol=1e-10, atol=1e-12), (j, b)
            assert np.allclose(sm[b][1], ref[1], rtol=1e-12)
    for b in range(2):
        for i in range(3):
            rows = _draft_rows_after_writeback(w, d, b, int(n_acc[b]), int(w.L[b]) + i + 1)
            ref = _dense_attention(d["x_q_mla"][b * 3 + i].double().numpy(), rows, scale)
            assert np.allclose(xo[(b, i)][0], ref[0], rtol=1e-10, atol=1e-12), (b, i)


# --------------------------------------------------------------------- paged / slotted KV

# page size 4; request 0 owns pages 2, 0, 5 (positions 0..11), request 1 pages 1, 3 and no third page
_BT = np.array([[2, 0, 5], [1, 3, -1]], dtype=np.int32)


def test_slot_of_hand_worked():
    assert paged.slot_of(_BT, 4, 0, 0) == 8        # page 2, offset 0
    assert paged.slot_of(_BT, 4, 0, 5) == 1        # page 0, offset 1
    assert paged.slot_of(_BT, 4, 0, 11) == 23      # page 5, offset 3
    assert paged.slot_of(_BT, 4, 1, 2) == 6        # page 1, offset 2
    assert paged.slot_of(_BT, 4, 1, 7) == 15       # page 3, offset 3
    assert paged.slot_of(_BT, 4, 1, 9) == -1       # no page
    assert paged.slot_of(_BT, 4, 1, -1) == -1
    assert paged.slot_of(_BT, 4, 0, 12) == -1      # past the table's three pages


def test_slot_of_page_size_one_is_the_token_table():
    req_to_token = np.array([[7, 3, 9, 0], [1, 2, 8, 5]], dtype=np.int32)
    for b in range(2):
        for s in range(4):
            assert paged.slot_of(req_to_token, 1, b, s) == req_to_token[b, s]


def test_assign_cache_locs_hand_worked():
    out = paged.assign_cache_locs(_BT, 4, [3, 1], 3)
    assert out.dtype == np.int64
    assert out.tolist() == [[11, 0, 1], [5, 6, 7]]   # request 0 crosses from page 2 into page 0


def test_paged_pool_built_page_by_page_reads_back_the_contiguous_cache():
    """A pool filled one page at a time from each request's page list (no slot
    arithmetic) holds, at slot_of(b, s), position s of the contiguous cache."""
    rng = np.random.default_rng(5)
    P, lengths = 8, [21, 8, 3]
    pages_needed = [(n + P - 1) // P for n in lengths]
    perm = rng.permutation(sum(pages_needed) + 2)        # pages handed out in a random order
    bt = np.full((3, max(pages_needed)), -1, dtype=np.int32)
    pool = np.full((len(perm) * P, 6), np.nan)
    cont = [rng.standard_normal((n, 6)) for n in lengths]
    k = 0
    for b, n in enumerate(lengths):
        for j in range(pages_needed[b]):
            page = int(perm[k]); k += 1
            bt[b, j] = page
            chunk = cont[b][j * P:(j + 1) * P]
            pool[page * P: page * P + len(chunk)] = chunk
    for b, n in enumerate(lengths):
        got = paged.gather_positions(pool, bt, P, b, range(n))
        assert np.array_equal(got, cont[b])
        got = paged.gather_positions(pool, bt, P, b, [n - 1, 0])
        assert np.array_equal(got, cont[b][[n - 1, 0]])


def test_kv_move_accepted_is_a_move_not_an_in_place_copy():
    """Window slots 10..13; the accepted rows are columns 1 and 0 (a swap):
    slot 10 receives slot 11's old bytes and slot 11 slot 10's old bytes.
    A copy done in place, in order, would leave both slots equal."""
    lat = np.arange(16 * 3, dtype=np.float32).reshape(16, 3)
    key = np.arange(16 * 2, dtype=np.uint8).reshape(16, 2)
    sc = np.arange(16, dtype=np.float32)
    loc = np.array([[10, 11, 12, 13]], dtype=np.int64)
    out = paged.kv_move_accepted([lat, key, sc], loc, np.array([[1, 0, -1, -1]]), [2])
    for before, after in zip([lat, key, sc], out):
        assert np.array_equal(after[10], before[11]) and np.array_equal(after[11], before[10])
        rest = [t for t in range(16) if t not in (10, 11)]
        assert np.array_equal(after[rest], before[rest])


def test_kv_move_accepted_hand_worked_shift_and_chain():
    lat = np.arange(20, dtype=np.float64).reshape(10, 2)
    loc = np.array([[2, 3, 4, 5], [6, 7, 8, 9]], dtype=np.int64)
    # request 0 keeps columns 1 and 3 (slots 3, 5) -> slots 2, 3; request 1 is a chain of 3
    (after,) = paged.kv_move_accepted([lat], loc, np.array([[1, 3, 0, 0], [0, 1, 2, 0]]), [2, 3])
    assert after[2].tolist() == lat[3].tolist() and after[3].tolist() == lat[5].tolist()
    assert np.array_equal(after[4:], lat[4:]) and np.array_equal(after[:2], lat[:2])
    # a chain (accept_index = 0, 1, 2, ...) moves nothing
    (same,) = paged.kv_move_accepted([lat], loc, np.tile(np.arange(4), (2, 1)), [4, 4])
    assert np.array_equal(same, lat)


def test_kv_writeback_slots_contiguous_special_case():
    """With dst_slots[b, i] = dst_start[b] + i the write-back by slot is the
    contiguous write-back."""
    rng = np.random.default_rng(9)
    B, Wn, T = 3, 4, 40
    sl = rng.standard_normal((B, Wn, 5)); sk = rng.integers(0, 256, (B, Wn, 7), dtype=np.uint8)
    ss = rng.standard_normal((B, Wn)).astype(np.float32)
    dl = rng.standard_normal((T, 5)); dk = rng.integers(0, 256, (T, 7), dtype=np.uint8)
    ds = rng.standard_normal(T).astype(np.float32)
    acc, start = [1, 4, 2], [0, 17, 30]
    slots = np.array([[start[b] + i for i in range(Wn)] for b in range(B)], dtype=np.int64)
    a = paged.kv_writeback_slots(sl, sk, ss, acc, dl, dk, ds, slots)
    e = writeback.kv_writeback(sl, sk, ss, acc, dl, dk, ds, start)
    for x, y in zip(a, e):
        assert np.array_equal(x, y)
    # scattered slots: row i lands where the plan says, nothing else changes
    slots = np.array([[39, 0, 5, 6], [12, 2, 31, 8], [20, 21, 1, 3]], dtype=np.int64)
    l2, k2, s2 = paged.kv_writeback_slots(sl, sk, ss, acc, dl, dk, ds, slots)
    touched = {int(slots[b, i]) for b in range(B) for i in range(acc[b])}
    for b in range(B):
        for i in range(acc[b]):
            t = int(slots[b, i])
            assert np.array_equal(l2[t], sl[b, i]) and np.array_equal(k2[t], sk[b, i]) and s2[t] == ss[b, i]
    rest = [t for t in range(T) if t not in touched]
    assert np.array_equal(l2[rest], dl[rest]) and np.array_equal(k2[rest], dk[rest])
