"""The device-side bounded wait gives up, flags the status word and leaves the
GPU usable.

Every mbarrier wait of the tensor-core kernels goes through one helper with a
2 s limit.  mtpsd_check_bounded_wait runs that helper, with a 1 ms limit, on a
barrier phase that nothing completes (two warps: CTA-scope and cluster-scope
acquire).  No fault, trap or endless loop is involved: the wait runs out, the
kernel returns, and a normal parity case runs right after on the same
context."""
import ctypes as C

import numpy as np
import pytest
import torch

from oracle import topk as otopk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def native():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mtp_speculative_decode_gb300 import _native
    _native.lib()
    return _native


def test_wait_runs_out_and_device_stays_usable(native):
    from mtp_speculative_decode_gb300 import api
    lib = native.lib()
    limit = 1_000_000   # 1 ms
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = torch.full((4,), -1, dtype=torch.int64, device="cuda")
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.mtpsd_check_bounded_wait(limit, C.c_void_p(status.data_ptr()), C.c_void_p(res.data_ptr()), stream)
    assert rc == 0, lib.mtpsd_last_error()
    torch.cuda.synchronize()
    r = res.cpu().numpy()
    assert status.item() & native.STATUS_WAIT_TIMEOUT
    assert r[1] == 0 and r[3] == 0, "both waits must give up"
    assert max(r[0], r[2]) >= limit, "the first wait to give up waited at least the limit"
    assert r[0] < 200 * limit and r[2] < 200 * limit, "neither wait ran far past the limit"

    # the context is intact: a top-k parity case runs right after
    rng = np.random.default_rng(3)
    R, V, k = 5, 9000, 2048
    sc = rng.normal(size=(R, V + 4)).astype(np.float32)
    lens = np.full(R, V, dtype=np.int64)
    got = api.topk(torch.from_numpy(sc).cuda(), torch.from_numpy(lens).cuda(), V, k).cpu().numpy()
    for i in range(R):
        assert np.array_equal(got[i], otopk.topk_select(sc[i, :V].astype(np.float64), k).astype(np.int32))
