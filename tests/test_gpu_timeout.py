"""The bounded-wait path on the GPU: a fused step whose first phase is never
reported complete (a completion threshold no launch reaches, set by a test
hook on the host) makes every projection that waits for it give up after the
wait limit.  The call reports WQ_ERR_TIMEOUT through the workspace's error
word, nothing faults, and the context stays usable: the same step then runs
normally and matches the oracle."""
import ctypes
import time

import numpy as np
import pytest
import torch

from wqtest import ARITH_TOL, REL_TOL, oracle_gemm, rel_err
from test_gpu_step import _descs, _layer_after, _uniform_stack

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def test_unreachable_dependency_times_out_and_the_context_survives():
    import weight_only_bit_wq_gb300 as wq
    projs = _uniform_stack(2, 4, 128, layers=1)
    after = _layer_after(len(projs))
    descs = _descs(wq, projs, after)
    ws = wq.new_step_workspace(descs, wq.WQ_STEP_FUSED)
    lib = wq._lib()
    lib.wq_internal_step_stall_probe.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                                 ctypes.c_size_t, ctypes.c_void_p]
    lib.wq_internal_step_stall_probe.restype = ctypes.c_int
    t0 = time.time()
    st = lib.wq_internal_step_stall_probe(ctypes.cast(descs, ctypes.c_void_p), len(descs),
                                          ctypes.c_void_p(ws.data_ptr()),
                                          ws.numel() * ws.element_size(), None)
    assert st == wq.WQ_OK
    with pytest.raises(wq.WQError) as e:
        wq.wq_check_workspace(ws)
    assert "abandoned" in str(e.value) or "TIMEOUT" in str(e.value).upper()
    assert time.time() - t0 < 60
    # the context is usable: a fresh workspace, the same step, the oracle's results
    wq.wq_workspace_init(ws)
    for p, w, x, d in projs:
        d["y"].fill_(float("nan"))
    wq.wq_step_run(descs, ws, flags=wq.WQ_STEP_FUSED)
    torch.cuda.synchronize()
    wq.wq_check_workspace(ws)
    for p, w, x, d in projs:
        err = rel_err(d["y"].cpu().numpy(), oracle_gemm(p, w, x))
        assert err <= REL_TOL and err <= ARITH_TOL, (p.name, err)
