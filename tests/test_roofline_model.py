"""The byte model used for the roofline reproduces the figures the pages
print (tests/golden/byte_model_from_pages.txt, each line cited there)."""
import os

from mtp_speculative_decode_gb300 import roofline

GOLD = os.path.join(os.path.dirname(__file__), "golden", "byte_model_from_pages.txt")
UNIT = {"GB": 1e9, "MB": 1e6, "B": 1.0}


def golden():
    out = {}
    for line in open(GOLD, encoding="utf-8"):
        if line.startswith("#") or not line.strip():
            continue
        name, value, unit, tol = line.split()
        out[name] = (float(value) * UNIT[unit], float(tol))
    return out


def close(got, want_tol):
    want, tol = want_tol
    return abs(got - want) <= tol * want + 1e-9


def test_page_figures():
    g = golden()
    K128, M1 = 128 * 1024, 1024 * 1024
    assert close(roofline.draft_indexer_read(K128, shared=False), g["draft_indexer_noshare_L128K"])
    assert close(roofline.draft_indexer_read(K128, shared=True), g["draft_indexer_share_L128K"])
    assert close(roofline.draft_indexer_read(M1, shared=False), g["draft_indexer_noshare_L1M"])
    assert close(roofline.draft_indexer_read(M1, shared=True), g["draft_indexer_share_L1M"])
    assert close(roofline.accepted_kv_move(32, 2.76, 78, 656), g["accepted_kv_move_b32"])
    # 656 = 512 FP8 latent + 16 bytes of scales + 64 bf16 rope values (the page gives only the total)
    assert close(512 + 16 + 64 * 2, g["kv_bytes_per_token_layer"])
    assert close(21 * 128, g["indexer_bytes_per_token_21L"])


def test_per_launch_models():
    # verify shape: 32 requests x 8192 context, 6 rows, 64 x 128 indexer heads
    vis_req = [8192 + 6] * 32
    vis_row = [8192 + i + 1 for i in range(6)] * 32
    assert roofline.indexer_flops(vis_row, 64, 128) == 2 * 64 * 128 * sum(vis_row)
    b = roofline.indexer_bytes(vis_req, 192, 64, 128)
    assert b == 32 * 8198 * 132 + 192 * 64 * 132 + 192 * 64 * 4
    assert roofline.mla_flops([2048] * 192, 128) == 192 * 2048 * 128 * 2 * 1088
