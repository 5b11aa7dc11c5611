"""The allocation-free indexer + top-k entry point (mtpsd_indexer_topk_noalloc).

Some callers cannot allocate device memory (a host whose allocator owns the
GPU memory, a serving loop that forbids allocation after start-up, a C caller
holding only raw input/output pointers); this entry point keeps its scratch in
a static device array of the library instead of a caller workspace.  The test
calls it through the C ABI twice in a row and checks each result against the
workspace entry point mtpsd_indexer_topk on the same inputs, with the tests'
criteria: top-k sets and order exact (index work), scores within 1e-2
relative; and, independently of that entry point, against the CPU oracle
(scores within 1e-2 relative, sets equal up to the 1e-4 tie band).  It also
checks that a call needing more scratch than the static maximum is refused
before any launch, and that a call whose score matrix would not fit runs when
the caller passes its own score buffer (the scratch then holds only the small
work plan).  Kept in a file that pytest collects last; it needs nothing from
the other tests."""
import ctypes as C

import numpy as np
import pytest
import torch

import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def native():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mtp_speculative_decode_gb300 import _native
    _native.lib()
    return _native


def _case(seed=11, lens=(3000, 8192, 100, 5000), r_per=6):
    rng = np.random.default_rng(seed)
    H, D, k = 64, 128, 2048
    lens = np.asarray(lens)
    B = len(lens)
    cap = lens + r_per + 2
    cache_start = np.concatenate([[0], np.cumsum(cap)[:-1]]).astype(np.int64)
    T = int(cap.sum())
    row_pos = (np.repeat(lens, r_per) + np.tile(np.arange(r_per), B)).astype(np.int64)
    R = len(row_pos)
    ro = np.arange(0, R + 1, r_per).astype(np.uint32)
    q = torch.from_numpy(rng.normal(size=(R, H, D)).astype(np.float32)).cuda()
    kx = torch.from_numpy(rng.normal(size=(T, D)).astype(np.float32)).cuda()
    w = torch.from_numpy(rng.uniform(0, 1, (R, H)).astype(np.float32)).cuda()
    return dict(H=H, D=D, k=k, B=B, R=R, q=q, kx=kx, w=w, cache_start=torch.from_numpy(cache_start).cuda(),
                ro=torch.from_numpy(ro).cuda(), row_pos=torch.from_numpy(row_pos).cuda(),
                maxv=int(row_pos.max()) + 1, h_cache_start=cache_start, h_row_pos=row_pos, r_per=r_per)


def _oracle_rows(c, rows):
    """Oracle scores of the given rows from the same float32 inputs (the
    oracle quantizes them with its own FP8 codec)."""
    from oracle import fp8 as ofp8
    from oracle import indexer as oindexer
    q = c["q"].cpu().numpy()
    kx = c["kx"].cpu().numpy()
    w = c["w"].cpu().numpy()
    out = {}
    for r in rows:
        b = r // c["r_per"]
        base = int(c["h_cache_start"][b])
        p = int(c["h_row_pos"][r])
        kc, ks = ofp8.quantize_block128(kx[base:base + p + 1])
        qc, qs = ofp8.quantize_block128(q[r])
        keys = ofp8.decode_e4m3(kc) * ks.astype(np.float64)
        qr = ofp8.decode_e4m3(qc) * qs.astype(np.float64)
        out[r] = oindexer.indexer_scores_row(qr, w[r], keys)
    return out


def _check_against_oracle(c, idx, sc, rows):
    ref = _oracle_rows(c, rows)
    for r in rows:
        parity.check_topk_row(idx[r], ref[r], c["k"])
        sel = idx[r][idx[r] >= 0]
        parity.check_scores_row(sc[r, :len(sel)], ref[r][sel])


def _args(native, c, qc, qs, kc, ks, idx, score, workspace=None, scores=None):
    return native.IndexerArgs(
        B=c["B"], R=c["R"], n_heads=c["H"], head_dim=c["D"], topk=c["k"], dtype=native.MTPSD_FP8_E4M3,
        q=qc.data_ptr(), q_scale=qs.data_ptr(), weights=c["w"].data_ptr(), k_cache=kc.data_ptr(),
        k_scale=ks.data_ptr(), pool_tokens=kc.shape[0], cache_start=c["cache_start"].data_ptr(),
        row_offsets=c["ro"].data_ptr(), row_pos=c["row_pos"].data_ptr(), max_visible=c["maxv"],
        topk_idx=idx.data_ptr(), topk_score=score.data_ptr(), scores=None if scores is None else scores.data_ptr(),
        workspace=None if workspace is None else workspace.data_ptr(),
        workspace_bytes=0 if workspace is None else workspace.numel(), dev_status=None)


def test_noalloc_matches_workspace_entry_point(native):
    from mtp_speculative_decode_gb300 import api
    lib = native.lib()
    c = _case()
    qc, qs = api.quantize_fp8_block128(c["q"])
    kc, ks = api.quantize_fp8_block128(c["kx"])
    qs = qs.reshape(c["R"], c["H"]).contiguous()
    ks = ks.reshape(-1).contiguous()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)

    ws = torch.empty(api.indexer_topk_workspace_size(c["B"], c["R"], c["maxv"], c["k"]), dtype=torch.uint8,
                     device="cuda")
    ref_idx = torch.empty(c["R"], c["k"], dtype=torch.int32, device="cuda")
    ref_sc = torch.empty(c["R"], c["k"], dtype=torch.float32, device="cuda")
    a = _args(native, c, qc, qs, kc, ks, ref_idx, ref_sc, ws)
    assert lib.mtpsd_indexer_topk(C.byref(a), stream) == 0, lib.mtpsd_last_error()
    torch.cuda.synchronize()
    ref_idx, ref_sc = ref_idx.cpu().numpy(), ref_sc.cpu().numpy()

    for call in range(2):   # two calls in a row share the static scratch
        idx = torch.full((c["R"], c["k"]), -7, dtype=torch.int32, device="cuda")
        sc = torch.zeros(c["R"], c["k"], dtype=torch.float32, device="cuda")
        a = _args(native, c, qc, qs, kc, ks, idx, sc, None)
        rc = lib.mtpsd_indexer_topk_noalloc(C.byref(a), stream)
        assert rc == 0, lib.mtpsd_last_error()
        torch.cuda.synchronize()
        idx, sc = idx.cpu().numpy(), sc.cpu().numpy()
        assert np.array_equal(idx, ref_idx), f"call {call}: top-k indices differ"
        for r in range(c["R"]):
            n = int((ref_idx[r] >= 0).sum())
            parity.check_scores_row(sc[r, :n], ref_sc[r, :n])
        # and against the oracle, independently of the workspace entry point
        _check_against_oracle(c, idx, sc, range(c["R"]))


def test_noalloc_with_caller_scores_beyond_the_static_maximum(native):
    """A score matrix of 48 rows x ~100k positions (19 MB) does not fit the
    16 MiB array; with the caller's score buffer only the work plan lives in
    the scratch, so the call runs and matches the oracle."""
    from mtp_speculative_decode_gb300 import api
    lib = native.lib()
    c = _case(seed=12, lens=(100000, 99000, 70000, 4000, 100001, 2500, 98000, 100000), r_per=6)
    ld = api.scores_ld(c["maxv"])
    assert c["R"] * ld * 4 > native.NOALLOC_SCRATCH_BYTES
    qc, qs = api.quantize_fp8_block128(c["q"])
    kc, ks = api.quantize_fp8_block128(c["kx"])
    qs = qs.reshape(c["R"], c["H"]).contiguous()
    ks = ks.reshape(-1).contiguous()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    # without a score buffer the call is refused before any launch
    idx = torch.full((c["R"], c["k"]), -7, dtype=torch.int32, device="cuda")
    sc = torch.zeros(c["R"], c["k"], dtype=torch.float32, device="cuda")
    a = _args(native, c, qc, qs, kc, ks, idx, sc, None)
    assert lib.mtpsd_indexer_topk_noalloc(C.byref(a), stream) == native.MTPSD_EWORKSPACE
    scores = torch.empty(c["R"], ld, dtype=torch.float32, device="cuda")
    for call in range(2):
        idx.fill_(-7)
        a = _args(native, c, qc, qs, kc, ks, idx, sc, None, scores=scores)
        rc = lib.mtpsd_indexer_topk_noalloc(C.byref(a), stream)
        assert rc == 0, lib.mtpsd_last_error()
        torch.cuda.synchronize()
        gi, gs = idx.cpu().numpy(), sc.cpu().numpy()
        _check_against_oracle(c, gi, gs, [0, 5, 26, c["R"] - 1])


def test_noalloc_rejects_oversize_before_launch(native):
    lib = native.lib()
    # 2048 rows x 1M positions of float32 scores is far beyond the static array
    a = native.IndexerArgs(B=1, R=2048, n_heads=64, head_dim=128, topk=2048, dtype=native.MTPSD_FP8_E4M3,
                           max_visible=1 << 20)
    rc = lib.mtpsd_indexer_topk_noalloc(C.byref(a), None)
    assert rc == native.MTPSD_EWORKSPACE
    assert b"static maximum" in lib.mtpsd_last_error()
