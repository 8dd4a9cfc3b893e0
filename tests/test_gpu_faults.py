"""The bounded pipeline waits, exercised without a fault: a test-only knob
lowers the wait limit to 1 ms and makes the production q4_K kernel withhold
the raw weight copy of its second super-block, so the waits for it run out.
The kernel must record MMQ_ERR_TIMEOUT, stop, drain what it issued, free its
tensor memory and return; the split-K tile counters must come back to zero;
and the next launches on the same stream must reproduce a clean run bit for
bit.  Nothing faults, traps or hangs: every wait gives up by itself."""
from __future__ import annotations

import ctypes
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from quantized_prefill_gemm_mmq_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_prefill_gemm_mmq_gb300 import ops as _ops
    from quantized_prefill_gemm_mmq_gb300 import _lib
    _lib.load()
    return _ops


def _status(lib):
    detail = (ctypes.c_int * 4)()
    st = lib.mmq_check_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), detail)
    return st, list(detail)


def test_bounded_wait_gives_up_and_the_next_launch_is_clean(ops):
    from quantized_prefill_gemm_mmq_gb300 import _lib
    lib = _lib.load()
    T, O, K = 256, 512, 1024
    w = torch.from_numpy(synth.make_weights("q4_K", O, K, 81)).cuda()
    x = torch.from_numpy(synth.make_x(T, K, 82, outliers=True)).cuda()
    _, ds, _, xa = ops.quantize_q8_1(x, want_qs=False, want_xh=False)
    ws = ops.SplitKWorkspace(xa.device, *ops.splitk_sizes(T, O, K, 2))
    clean = ops.gemm("q4_K", w, xa, ds, O)
    clean_sk = ops.gemm_splitk(w, xa, ds, O, ksplit=2, workspace=ws)
    assert _status(lib) == (0, [0, 0, 0, 0])
    try:
        assert lib.mmq_debug_fault_inject(1, 1000) == 0          # withhold a copy; 1 ms wait limit
        t0 = time.perf_counter()
        ops.gemm("q4_K", w, xa, ds, O)
        st, detail = _status(lib)
        assert st == -5 and detail[0] == -5                      # MMQ_ERR_TIMEOUT
        assert detail[1] == 9                                    # the production q4_K kernel
        assert 1 <= detail[2] <= 11                              # a recorded wait site
        assert time.perf_counter() - t0 < 10.0                   # it gave up on its own
        info = (ctypes.c_int * 4)()
        assert lib.mmq_last_failure_info(info) == 0 and info[0] >= 1000   # waited at least the 1 ms limit (us)
        ops.gemm_splitk(w, xa, ds, O, ksplit=2, workspace=ws)
        st, detail = _status(lib)
        assert st == -5 and detail[1] == 9
        assert int(ws.counters.abs().sum()) == 0                 # every tile counter back at zero
    finally:
        assert lib.mmq_debug_fault_inject(0, 0) == 0
    assert _status(lib) == (0, [0, 0, 0, 0])                     # the status word was cleared
    again = ops.gemm("q4_K", w, xa, ds, O)
    again_sk = ops.gemm_splitk(w, xa, ds, O, ksplit=2, workspace=ws)
    assert _status(lib)[0] == 0
    assert torch.equal(again, clean) and torch.equal(again_sk, clean_sk)
    assert int(ws.counters.abs().sum()) == 0
    assert np.isfinite(again.cpu().numpy()).all()
