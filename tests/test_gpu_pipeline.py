"""End-to-end parity of the decode step (merge, verify indexer + top-k +
sparse MLA, acceptance, write-back, shared-index draft loop) on the five
workloads: every output for the tiny one, sampled rows at full size."""
import numpy as np
import pytest
import torch

import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mtp_speculative_decode_gb300 import _native, pipeline, workloads
    from oracle.pipeline import OracleStep
    _native.lib()
    return pipeline, workloads, OracleStep


def _sample(n, k, seed):
    rng = np.random.default_rng(seed)
    return sorted(set([0, n - 1] + list(rng.choice(n, size=min(n, k), replace=False))))


def run_case(mods, name, n_rows, n_reqs, heads=None, latent_fp8=False, page_size=None):
    pipeline, W, OracleStep = mods
    w = W.build(name)
    d = W.draft_tensors(w) if w.spec.draft_steps else None
    g = pipeline.DecodeStep(w, "cuda", d, latent_fp8=latent_fp8, page_size=page_size)
    g.step()
    torch.cuda.synchronize()
    assert g.status.item() == 0, f"device status {g.status.item()}"
    o = OracleStep(w, d, latent_fp8=latent_fp8)
    spec = w.spec
    tol = parity.ATT_TOL_F32 if spec.latent_f32 else parity.ATT_TOL_BF16
    report = {}
    if spec.verify:
        mt, mo = o.merge()
        assert np.array_equal(g.merged_tokens.cpu().numpy(), mt)
        assert np.array_equal(g.merged_offsets.cpu().numpy().astype(np.int64), mo.astype(np.int64))
        rows = _sample(w.R, n_rows, 1)
        sc = o.verify_scores(rows)
        tk = o.verify_topk(sc)
        gi = g.topk_idx.cpu().numpy()
        diffs = {r: parity.check_topk_row(gi[r], sc[r], spec.topk) for r in rows}
        report["topk_tie_diffs"] = sum(diffs.values())
        # a near-tie resolved the other way (within the band) leaves two correct selections:
        # the production output is then checked against the oracle's attention over the
        # GPU's own selection
        sel = {r: (gi[r] if diffs[r] else tk[r]) for r in rows}
        ref = o.verify_mla(sel, heads=heads)
        go = g.out.float().cpu().numpy()
        errs = []
        for r in rows:
            gr = go[r] if heads is None else go[r][list(heads)]
            errs.append(parity.check_attention_row(gr, ref[r][0], tol))
        report["verify_att_err"] = max(errs)
    n_acc, nxt = o.accept()
    assert np.array_equal(g.num_accepted.cpu().numpy(), n_acc)
    assert np.array_equal(g.next_tokens.cpu().numpy(), nxt)
    if spec.draft_steps:
        P = o.next_pos(n_acc)
        assert np.array_equal(g.next_pos.cpu().numpy(), P)
        reqs = _sample(w.B, n_reqs, 2)
        s0sc, s0 = o.draft_step0(n_acc, reqs)
        gd = g.d_topk.cpu().numpy()
        gs = g.shared_idx.cpu().numpy()
        report["draft_tie_diffs"] = sum(parity.check_topk_row(gd[b], s0sc[b], spec.topk) for b in reqs)
        assert np.array_equal(gs, gd)                 # one step-0 row per request: the share is that row
        ddiffs = {b: parity.check_topk_row(gd[b], s0sc[b], spec.topk) for b in reqs}
        errs = []
        # the oracle attends over its own step-0 selection, or over the GPU's where the two
        # differ only within the tie band
        sel = {b: (gd[b] if ddiffs[b] else s0[b]) for b in reqs}
        for j in range(spec.draft_steps):
            ref = o.draft_mla(n_acc, sel, j, reqs, heads=heads)
            go = g.d_out[j].float().cpu().numpy()
            for b in reqs:
                gr = go[b] if heads is None else go[b][list(heads)]
                errs.append(parity.check_attention_row(gr, ref[b][0], tol))
        report["draft_att_err"] = max(errs)
    print(name, report)
    return report


def test_tiny_all_rows(mods):
    run_case(mods, "tiny", n_rows=10 ** 6, n_reqs=10 ** 6)


@pytest.mark.parametrize("ps", [4, 64])
def test_tiny_paged(mods, ps):
    """The step over paged caches (shuffled pages, one block table for both layers): the slot plan, the
    accepted-KV move and the write-back by slot, and every read through the table, give the contiguous
    step's results against the oracle.  The paged pools hold the workload's caches where the oracle's slot
    map says, before and after the step."""
    from oracle import paged as opaged
    pipeline, W, _ = mods
    run_case(mods, "tiny", n_rows=10 ** 6, n_reqs=10 ** 6, page_size=ps)
    w = W.build("tiny")
    g = pipeline.DecodeStep(w, "cuda", W.draft_tensors(w), page_size=ps)
    bt = g.block_table_host
    lat = g.latent.cpu().numpy()
    for b in range(w.B):
        pos = range(int(w.L[b]) + w.r)
        got = opaged.gather_positions(lat, bt, ps, b, pos)
        want = np.asarray(w.tensors["latent"])[int(w.cache_start[b]) + np.arange(len(pos))]
        assert np.array_equal(got, want)
    g.step()
    torch.cuda.synchronize()
    assert g.status.item() == 0
    want_loc = opaged.assign_cache_locs(bt, ps, w.L, w.spec.K + 1)
    assert np.array_equal(g.out_cache_loc.cpu().numpy(), want_loc)


@pytest.mark.slow
def test_verify_paged_full_size(mods):
    run_case(mods, "verify", n_rows=16, n_reqs=6, heads=range(0, 128, 16), page_size=64)


@pytest.mark.slow
def test_draft_loop_paged_full_size(mods):
    run_case(mods, "draft", n_rows=0, n_reqs=6, heads=range(0, 128, 16), page_size=64)


@pytest.mark.slow
def test_verify_full_size(mods):
    run_case(mods, "verify", n_rows=24, n_reqs=0, heads=None)


@pytest.mark.slow
def test_draft_loop_full_size(mods):
    run_case(mods, "draft", n_rows=0, n_reqs=8)


@pytest.mark.slow
def test_long_context_full_size(mods):
    run_case(mods, "long", n_rows=4, n_reqs=0)


@pytest.mark.slow
def test_draft_loop_fp8_latent(mods):
    """The draft loop (write-back, step-0 indexer, four shared-index MLA steps) over 656-byte FP8 latent rows."""
    run_case(mods, "draft", n_rows=0, n_reqs=6, heads=range(0, 128, 16), latent_fp8=True)


@pytest.mark.slow
def test_verify_fp8_latent(mods):
    run_case(mods, "verify", n_rows=12, n_reqs=4, heads=range(0, 128, 16), latent_fp8=True)


@pytest.mark.slow
def test_decode_step_full_size(mods):
    run_case(mods, "decode", n_rows=10, n_reqs=6, heads=range(0, 128, 8))


# ----------------------------------------------------------------------------- cross-layer and cross-phase reuse

def run_layered(mods, name, types, n_rows, heads=None):
    """A multi-layer verify with the full/shared indexer schedule against the oracle."""
    pipeline, W, OracleStep = mods
    w = W.add_layers(W.build(name), len(types))
    g = pipeline.LayeredVerify(w, types, "cuda")
    g.step()
    torch.cuda.synchronize()
    assert g.status.item() == 0, f"device status {g.status.item()}"
    o = OracleStep(w)
    k = w.spec.topk
    tol = parity.ATT_TOL_F32 if w.spec.latent_f32 else parity.ATT_TOL_BF16
    rows = _sample(w.R, n_rows, 3)
    used, errs, ties = {}, [], 0
    for l, typ in enumerate(types):
        L = g.layers[l]
        if typ == "full":
            sc = o.verify_scores(rows, layer=l)
            tk = o.verify_topk(sc)
            gi = L["topk"].cpu().numpy()
            diffs = {r: parity.check_topk_row(gi[r], sc[r], k) for r in rows}
            ties += sum(diffs.values())
            used[l] = {r: (gi[r] if diffs[r] else tk[r]) for r in rows}
        ref = o.verify_mla(used[L["src"]], heads=heads, layer=l)
        go = L["out"].float().cpu().numpy()
        for r in rows:
            gr = go[r] if heads is None else go[r][list(heads)]
            errs.append(parity.check_attention_row(gr, ref[r][0], tol))
    print(name, types, {"tie_diffs": ties, "att_err": max(errs)})


def test_layered_verify_tiny(mods):
    run_layered(mods, "tiny", ["full", "shared", "full", "shared"], n_rows=10 ** 6)


@pytest.mark.slow
def test_layered_verify_full_size(mods):
    run_layered(mods, "verify", ["full", "shared", "shared", "shared"], n_rows=12, heads=range(0, 128, 16))


def run_seeded(mods, name, n_reqs, heads=None):
    """draft_extend's attention over the window rows, the seed gathered at the last accepted row, and the
    next round's draft steps over the seed plus the new positions, against the oracle."""
    pipeline, W, OracleStep = mods
    w = W.add_draft_extend(W.build(name))
    d = W.draft_tensors(w)
    g = pipeline.DecodeStep(w, "cuda", d, seeded=True)
    g.step()
    torch.cuda.synchronize()
    assert g.status.item() == 0, f"device status {g.status.item()}"
    o = OracleStep(w, d)
    k, Wn = w.spec.topk, w.spec.K + 1
    tol = parity.ATT_TOL_F32 if w.spec.latent_f32 else parity.ATT_TOL_BF16
    n_acc, _ = o.accept()
    assert np.array_equal(g.num_accepted.cpu().numpy(), n_acc)
    reqs = _sample(w.B, n_reqs, 4)
    gx = g.x_topk.cpu().numpy()
    sc, tk, _ = o.draft_extend(n_acc, reqs, heads=heads)
    diffs = {(b, i): parity.check_topk_row(gx[b * Wn + i], sc[(b, i)], k) for b in reqs for i in range(Wn)}
    chosen = {key: (gx[key[0] * Wn + key[1]] if diffs[key] else tk[key]) for key in diffs}
    _, _, ref = o.draft_extend(n_acc, reqs, heads=heads, selections=chosen)
    gxo = g.x_out.float().cpu().numpy()
    errs = []
    for (b, i), (o_ref, _) in ref.items():
        gr = gxo[b * Wn + i] if heads is None else gxo[b * Wn + i][list(heads)]
        errs.append(parity.check_attention_row(gr, o_ref, tol))
    # the seed is the selection of row num_accepted, at position L + num_accepted (exact)
    gs = g.shared_idx.cpu().numpy()
    gsp = g.seed_pos.cpu().numpy()
    for b in range(w.B):
        assert np.array_equal(gs[b], gx[b * Wn + n_acc[b]])
        assert gsp[b] == w.L[b] + n_acc[b]
    seed = {b: chosen[(b, int(n_acc[b]))] for b in reqs}
    for j in range(w.spec.draft_steps):
        ref = o.seeded_draft_mla(n_acc, seed, j, reqs, heads=heads)
        go = g.d_out[j].float().cpu().numpy()
        for b in reqs:
            gr = go[b] if heads is None else go[b][list(heads)]
            errs.append(parity.check_attention_row(gr, ref[b][0], tol))
    print(name, "seeded", {"tie_diffs": sum(diffs.values()), "att_err": max(errs)})


def test_seeded_draft_tiny(mods):
    run_seeded(mods, "tiny", n_reqs=10 ** 6)


@pytest.mark.slow
def test_seeded_draft_full_size(mods):
    run_seeded(mods, "draft", n_reqs=4, heads=range(0, 128, 16))
