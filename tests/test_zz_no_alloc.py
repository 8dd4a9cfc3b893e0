"""The split-K q4_K GEMM on the library's static scratch against the
caller-workspace entry point.  For callers that cannot allocate device memory
(an allocator-less host runtime, code running while device allocation is not
allowed): the entry point itself allocates nothing, which the tests check
through the CUDA free-memory count and torch's allocator.  Kept in a file of
its own that is collected last: it must pass alone and after every other test
(the static counters carry over between calls)."""
from __future__ import annotations

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


@pytest.mark.parametrize("T,O,K,ksplit", [(16, 4096, 4096, 4), (64, 4096, 11008, 4), (130, 300, 1280, 3),
                                          (1, 128, 2816, 11), (200, 256, 768, 1)])
def test_static_scratch_matches_caller_workspace(ops, T, O, K, ksplit):
    w = torch.from_numpy(synth.make_weights("q4_K", O, K, seed=T + O + K)).cuda()
    x = torch.from_numpy(synth.make_x(T, K, seed=O + 5, outliers=True)).cuda()
    _, ds, _, xa = ops.quantize_q8_1(x, want_qs=False, want_xh=False)
    ref = ops.gemm_splitk(w, xa, ds, O, ksplit=ksplit)
    a = torch.empty_like(ref)
    b = torch.empty_like(ref)
    ops.gemm_splitk_static(w, xa, ds, O, ksplit=ksplit, out=a)   # first call: the library's one-time set-up
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    ops.gemm_splitk_static(w, xa, ds, O, ksplit=ksplit, out=a)
    ops.gemm_splitk_static(w, xa, ds, O, ksplit=ksplit, out=b)   # two calls in a row: counters were reset
    ops.check_status()
    assert torch.cuda.mem_get_info()[0] == free0                 # no device memory taken by the calls
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.equal(a, ref)
    assert torch.equal(b, ref)


def test_static_scratch_refuses_oversize(ops):
    from quantized_prefill_gemm_mmq_gb300._lib import MMQError
    T, O, K = 2048, 4096, 4096     # 4 splits x 2048 x 4096 f32 = 128 MiB > 16 MiB of static scratch
    w = torch.zeros(O * (K // 256) * 144, dtype=torch.uint8, device="cuda")
    xa = torch.zeros((2, T, K), dtype=torch.float16, device="cuda")
    ds = torch.zeros((T, K // 32), dtype=torch.int32, device="cuda")
    with pytest.raises(MMQError) as e:
        ops.gemm_splitk_static(w, xa, ds, O, ksplit=4)
    assert e.value.status == -9
    y = ops.gemm_splitk_static(w[: 128 * (K // 256) * 144], xa[:, :16].contiguous(), ds[:16].contiguous(), 128,
                               ksplit=4)
    ops.check_status()
    assert torch.equal(y, torch.zeros_like(y))
