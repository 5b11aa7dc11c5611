"""The C-ABI library loads and exports every symbol include/mtpsd.h declares,
the ctypes structures match the C layout, and host-side argument checks
reject bad calls before any launch.  CPU only (no compute call)."""
import ctypes as C
import os
import re
import subprocess
import tempfile

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mtpsd.h")


@pytest.fixture(scope="module")
def native():
    from mtp_speculative_decode_gb300 import _native
    if not os.path.exists(_native.LIB_PATH):
        from mtp_speculative_decode_gb300 import build
        build.build()
    _native.lib()
    return _native


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mtpsd_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(native):
    names = declared_functions()
    assert len(names) >= 14
    lib = native.lib()
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
        assert n in native.SIGNATURES, f"{n} has no ctypes signature"
    assert set(native.SIGNATURES) == set(names)


def _c_offsets(struct, fields):
    src = "#include <stddef.h>\n#include <stdio.h>\n#include \"mtpsd.h\"\nint main(void){\n"
    src += f'printf("%zu\\n", sizeof({struct}));\n'
    for f in fields:
        src += f'printf("%zu\\n", offsetof({struct}, {f}));\n'
    src += "return 0;}\n"
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "t.c")
        exe = os.path.join(d, "t")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-I", os.path.dirname(HEADER), c, "-o", exe], check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.split()
    return [int(x) for x in out]


@pytest.mark.parametrize("cname,pyname", [("mtpsd_indexer_args", "IndexerArgs"), ("mtpsd_mla_args", "MlaArgs"),
                                          ("mtpsd_paged_kv", "PagedKV")])
def test_struct_layout_matches_header(native, cname, pyname):
    st = getattr(native, pyname)
    fields = [f for f, _ in st._fields_]
    got = _c_offsets(cname, fields)
    assert got[0] == C.sizeof(st)
    assert got[1:] == [getattr(st, f).offset for f in fields]


def test_host_checks_reject_before_launch(native):
    lib = native.lib()
    assert lib.mtpsd_merge_tokens(None, 0, None, None, 0, 0, None, None, None) == native.MTPSD_EINVAL
    assert b"B >= 1" in lib.mtpsd_last_error()
    assert lib.mtpsd_accept_greedy(None, None, -1, 0, -1, None, None, None) == native.MTPSD_EINVAL
    a = native.IndexerArgs(B=1, R=1, n_heads=64, head_dim=64, topk=16, dtype=native.MTPSD_FP8_E4M3)
    assert lib.mtpsd_indexer_topk(C.byref(a), None) == native.MTPSD_EUNSUPPORTED
    a = native.IndexerArgs(B=1, R=1, n_heads=64, head_dim=128, topk=16, dtype=native.MTPSD_FP8_E4M3,
                           q=1, q_scale=1, weights=1, k_cache=1, k_scale=1, cache_start=1, row_offsets=1,
                           row_pos=1, topk_idx=1, max_visible=100)
    assert lib.mtpsd_indexer_topk(C.byref(a), None) == native.MTPSD_EWORKSPACE
    m = native.MlaArgs(B=1, R=1, n_heads=128, d_latent=512, d_v=512, n_idx=16, dtype=native.MTPSD_BF16)
    assert lib.mtpsd_sparse_mla_decode(C.byref(m), None) == native.MTPSD_EUNSUPPORTED
    m = native.MlaArgs(B=1, R=1, n_heads=20, d_latent=576, d_v=512, n_idx=16, dtype=native.MTPSD_BF16)
    assert lib.mtpsd_sparse_mla_decode(C.byref(m), None) == native.MTPSD_EUNSUPPORTED
    m = native.MlaArgs(B=1, R=1, n_heads=16, d_latent=576, d_v=512, n_idx=16, n_append=2,
                       dtype=native.MTPSD_BF16)
    assert lib.mtpsd_sparse_mla_decode(C.byref(m), None) == native.MTPSD_EINVAL
    assert lib.mtpsd_kv_writeback(None, None, None, 1, 6, 7, 128, None, None, None, None, None, None, 10, None,
                                  None, None) == native.MTPSD_EUNSUPPORTED
    assert lib.mtpsd_topk(None, 10, 1, None, 0, 20, 4, None, None, None, 0, None, None) == native.MTPSD_EINVAL
    assert lib.mtpsd_check_bounded_wait(0, 8, 8, None) == native.MTPSD_EINVAL
    assert lib.mtpsd_check_bounded_wait(2_000_000_000, 8, 8, None) == native.MTPSD_EINVAL
    assert lib.mtpsd_check_bounded_wait(1000, None, 8, None) == native.MTPSD_EINVAL


def test_paged_checks_reject_before_launch(native):
    lib = native.lib()
    m = native.MlaArgs(B=1, R=1, n_heads=16, d_latent=576, d_v=512, n_idx=16, dtype=native.MTPSD_BF16)
    for ps, bt, stride in ((3, 8, 4), (0, 8, 4), (1 << 17, 8, 4), (64, None, 4), (64, 8, 0)):
        pk = native.PagedKV(block_table=bt, bt_stride=stride, page_size=ps)
        assert lib.mtpsd_sparse_mla_decode_paged(C.byref(m), C.byref(pk), None) == native.MTPSD_EINVAL
        assert b"page" in lib.mtpsd_last_error() or b"block_table" in lib.mtpsd_last_error()
        assert lib.mtpsd_assign_cache_locs(C.byref(pk), 1, 8, 4, 8, None, None) == native.MTPSD_EINVAL
    a = native.IndexerArgs(B=1, R=1, n_heads=64, head_dim=128, topk=16, dtype=native.MTPSD_FP8_E4M3)
    pk = native.PagedKV(block_table=8, bt_stride=4, page_size=48)
    assert lib.mtpsd_indexer_topk_paged(C.byref(a), C.byref(pk), None) == native.MTPSD_EINVAL
    assert lib.mtpsd_assign_cache_locs(None, 1, 8, 4, 8, None, None) == native.MTPSD_EINVAL
    # window wider than the move's shared staging, and an unknown latent type
    assert lib.mtpsd_kv_move_accepted(8, native.MTPSD_BF16, None, 0, None, 10, 8, 8, 8, 1, 17, None,
                                      None) == native.MTPSD_EINVAL
    assert lib.mtpsd_kv_move_accepted(8, 7, None, 0, None, 10, 8, 8, 8, 1, 4, None, None) == native.MTPSD_EUNSUPPORTED
    assert lib.mtpsd_kv_writeback_slots(None, None, None, 1, 6, native.MTPSD_BF16, 128, None, None, None, None, None,
                                        10, None, None, None, None) == native.MTPSD_EINVAL
    assert lib.mtpsd_kv_writeback_slots(16, 16, None, 1, 6, native.MTPSD_BF16, 128, 8, 16, 16, None, 8,
                                        10, 8, None, None, None) == native.MTPSD_EINVAL   # dst_pos without next_pos


def test_host_merged_offsets_mirror(native):
    from mtp_speculative_decode_gb300 import host_merged_offsets
    from oracle import merge as omerge
    rng = np.random.default_rng(0)
    for K in (0, 1, 5):
        po = np.concatenate([[0], np.cumsum(rng.integers(0, 4, 30))]).astype(np.uint32)
        assert np.array_equal(host_merged_offsets(po, K), omerge.host_merged_offsets(po, K))


def test_workspace_queries(native):
    lib = native.lib()
    assert lib.mtpsd_scores_ld(8198) % 4 == 0 and lib.mtpsd_scores_ld(8198) >= 8198
    ws = lib.mtpsd_indexer_topk_workspace_size(32, 192, 8198, 2048)
    assert ws >= 192 * 8198 * 4
    assert lib.mtpsd_topk_workspace_size(192, 40960, 2048) == 0
    # split path: two list buffers of 8-byte entries (16384-key segments; 100000 keys: level 1 has 7 lists
    # of 2048, level 2 is final; 600000 keys: 37 lists, then 5, then the final one)
    assert lib.mtpsd_topk_workspace_size(10, 100000, 2048) == 10 * 7 * 2048 * 8
    assert lib.mtpsd_topk_workspace_size(10, 600000, 2048) == 10 * 37 * 2048 * 8 + 10 * 5 * 2048 * 8
    plan = lib.mtpsd_indexer_topk_plan_bytes(32, 192)
    assert 0 < plan < 64 * 1024 and plan % 256 == 0
    # the workspace is the padded score matrix followed by the plan
    assert ws == (192 * lib.mtpsd_scores_ld(8198) * 4 + 255) // 256 * 256 + plan


def test_launch_count_queries(native):
    """The launch-count queries answer on any machine (without a device they describe the portable
    kernels): nothing for an empty call, one or two launches otherwise."""
    lib = native.lib()
    assert lib.mtpsd_sparse_mla_launch_count(0, 128, 2048, 0, native.MTPSD_BF16) == 0
    for R, n_append in ((192, 0), (32, 3), (1, 0)):
        assert lib.mtpsd_sparse_mla_launch_count(R, 128, 2048, n_append, native.MTPSD_BF16) in (1, 2)
        assert lib.mtpsd_sparse_mla_launch_count(R, 128, 2048, n_append, native.MTPSD_F32) in (1, 2)
    assert lib.mtpsd_indexer_topk_launch_count(64, 128, native.MTPSD_FP8_E4M3, 8198, 2048) in (2, 3)
    assert lib.mtpsd_indexer_topk_launch_count(64, 128, native.MTPSD_F32, 8198, 2048) == 2
    assert lib.mtpsd_indexer_topk_launch_count(48, 128, native.MTPSD_FP8_E4M3, 8198, 2048) == 2   # no tensor-core shape
    # rows past 40960 keys: one launch per split level (16384-key segments, then merges of 8 lists of 2048)
    assert lib.mtpsd_topk_launch_count(40960, 2048) == 1
    assert lib.mtpsd_topk_launch_count(40961, 2048) == 2
    assert lib.mtpsd_topk_launch_count(8 * 16384, 2048) == 2
    assert lib.mtpsd_topk_launch_count(8 * 16384 + 1, 2048) == 3
    assert lib.mtpsd_topk_launch_count(1 << 20, 4096) == 4            # 64 segments, merges of 4: 16, 4, 1
    assert lib.mtpsd_indexer_topk_launch_count(48, 128, native.MTPSD_F32, 100000, 2048) == 3


def test_indexer_schedule_matches_the_oracle(native):
    from mtp_speculative_decode_gb300 import api
    from oracle import share
    cases = [dict(n_layers=78, freq=4, offset=2), dict(n_layers=3), dict(n_layers=4, pattern="FSSF"),
             dict(n_layers=5, freq=1), dict(n_layers=6, freq=2, offset=1), dict(n_layers=9, offset=4),
             dict(n_layers=7, freq=3), dict(n_layers=0)]
    for c in cases:
        assert api.resolve_indexer_types(**c) == share.resolve_indexer_types(**c), c
    for bad in (dict(n_layers=3, pattern="SFF"), dict(n_layers=3, pattern="FX"), dict(n_layers=2, pattern="FFF")):
        with pytest.raises(Exception):
            api.resolve_indexer_types(**bad)
