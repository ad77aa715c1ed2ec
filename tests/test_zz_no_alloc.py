"""The decode entry point that allocates nothing.

kvq_decode_static_scratch serves callers that cannot call cudaMalloc on their
decode path (for example an operator embedded in a runtime that owns every
device allocation, or a loop that cannot afford the synchronisation an
allocation implies).  Its scratch is a fixed device array inside the library,
so the test checks that it gives the same results as kvq_decode with a caller
workspace, on two calls in a row (the second call sees the array the first
one left behind), and that an oversized request is refused before any launch.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest

from harness import DeviceRun, small_workload
from synth import make_inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)


@pytest.mark.parametrize("fmt", [dict(k_bits=8, v_bits=8, window=32), dict(k_bits=4, v_bits=8, q_heads=32),
                                 dict(k_bits=4, v_bits=4, asym=True, q_bits=8)])
def test_static_scratch_matches_workspace_decode_on_two_calls(fmt):
    kw = dict(batch=5, q_heads=16, kv_heads=4, len_range=(1, 400))
    kw.update(fmt)
    inp = make_inputs(small_workload("no_alloc", **kw))
    run = DeviceRun(inp)
    lib = run.lib
    w = inp.workload
    ref, ref_lse = run.decode(out_fp32=True)
    for call in range(2):
        out = torch.full((w.batch, w.q_heads, 128), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((w.batch, w.q_heads), float("nan"), dtype=torch.float32, device="cuda")
        lib.kvq_decode_static_scratch(run.cache.desc, run.q, w.batch, w.q_heads, run.lens, run.table,
                                      inp.max_blocks, out, lse=lse, err_word=run.err)
        torch.cuda.synchronize()
        o, l = out.cpu().numpy(), lse.cpu().numpy()
        assert np.all(np.isfinite(o)), f"call {call}: non-finite output"
        # same kernel, same plan and a fixed merge order: the results are the
        # workspace call's bit for bit, so any trace of the previous call's
        # scratch contents would show
        np.testing.assert_array_equal(o, ref, err_msg=f"call {call}")
        np.testing.assert_array_equal(l, ref_lse, err_msg=f"call {call}")
    assert run.err_bits() == 0


def test_static_scratch_refuses_plans_beyond_its_size():
    inp = make_inputs(small_workload("no_alloc_big", batch=2, len_range=(20, 40)))
    run = DeviceRun(inp)
    lib = run.lib
    big_batch, q_heads = 4096, 8               # 8192 units: far more scratch than the fixed array holds
    plan = lib.kvq_decode_device_plan(run.cache.desc, big_batch, q_heads)
    assert plan.workspace_bytes > lib.STATIC_SCRATCH_BYTES
    out = torch.zeros((2, 8, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(lib.KvqError) as e:
        lib.kvq_decode_static_scratch(run.cache.desc, run.q, big_batch, q_heads, run.lens, run.table,
                                      inp.max_blocks, out)
    assert e.value.status == lib.KVQ_ERR_WORKSPACE
