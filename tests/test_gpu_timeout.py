"""Device-side failure detection without a GPU fault: every wait in the skinny kernel is bounded
(ql_set_wait_limit).  With the limit at 0 the producer gives up on the activation hand-off at its
first poll, flags QL_DEV_TIMEOUT in the workspace status word, still issues its loads (so no
stage is left waiting) and the kernel returns; the host reads the flag, re-initialises the
workspace and the next call is exact again.  No wait here is unbounded and nothing traps."""
import numpy as np
import pytest
import torch

import synth
from _util import gpu_lib, to_bf16_tensor
from oracle import qlinear_oracle as Q

pytestmark = pytest.mark.gpu

DEV_TIMEOUT = 1
DEFAULT_WAIT_LIMIT = 1 << 20


@pytest.fixture(scope="module")
def ql():
    return gpu_lib()


def test_wait_timeout_is_reported_and_recoverable(ql):
    c = synth.int8_case(2, 640, 2048, seed=7)
    x = to_bf16_tensor(c["x"])
    w = torch.from_numpy(c["w"]).cuda()
    s = torch.from_numpy(c["w_s"]).cuda()
    ref = Q.int8_w8a8(c["x"], c["w"], c["w_s"])
    ws = ql.Workspace()

    def call():
        _, acc, _, _, _ = ql.qlinear_int8_w8a8(x, w, s, debug=True, workspace=ws)
        torch.cuda.synchronize()
        return acc.cpu().numpy()

    assert np.array_equal(call(), ref["acc"])
    st, flags = ql.read_device_status(ws.buf)
    assert st == 0 and flags == 0

    ql.set_wait_limit(0)
    try:
        seen = False
        for _ in range(8):  # the first poll finds the image unfinished in practice; retry to be sure
            call()
            st, flags = ql.read_device_status(ws.buf, clear=True)
            if flags & DEV_TIMEOUT:
                seen = True
                break
    finally:
        ql.set_wait_limit(DEFAULT_WAIT_LIMIT)
    assert seen, "a zero wait limit never timed out"
    assert st != 0  # read_device_status reports QL_ERR_TIMEOUT with the flag

    # the context survives: counters may be left mid-count, so re-initialise the workspace
    ws.buf.zero_()
    torch.cuda.synchronize()
    assert np.array_equal(call(), ref["acc"])
    st, flags = ql.read_device_status(ws.buf)
    assert st == 0 and flags == 0
