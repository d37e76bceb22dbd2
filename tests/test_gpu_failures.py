"""Failure detection without a GPU fault.

A wait that nothing satisfies must end in an error status the host can read,
with the context still usable; an allocation that cannot succeed must come
back as OUT_OF_MEMORY with the handle still usable.  Nothing here traps,
faults or hangs the GPU: the wait is bounded (tens of milliseconds) and the
failed allocation is refused by the driver before any memory is touched.
"""
import numpy as np
import pytest

import oracle
import synthetic

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def q4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gptq_bit_weight_gb300 as q4mod
    return q4mod


def to_dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def check_layer_still_works(q4, mat, layer, K, N, gs):
    dq = oracle.dequantize_layer(layer.qweight, layer.qzeros, layer.scales, layer.g_idx, K, N, gs)
    x = synthetic.activations(3, K, key=(91, K, N))
    y = mat(to_dev(x))
    torch.cuda.synchronize()
    y_ref = oracle.reference_output(x, dq, layer.bias)
    tol = oracle.tolerance(x, dq.w16, y_ref, K)
    assert np.all(np.abs(y.float().cpu().numpy().astype(np.float64) - y_ref) <= tol)
    mat.device_error()


def test_bounded_wait_runs_out_and_reports(q4):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    q4.gptq_q4_debug_wait_probe(status.data_ptr(), 20000, stream.cuda_stream)   # 20 ms limit
    b.record(stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    ms = a.elapsed_time(b)
    assert 15.0 <= ms < 1000.0, ms
    # the context is intact: an ordinary layer still computes the right answer
    K, N, gs = 512, 256, 128
    layer = synthetic.make_layer(K, N, gs, bias=True, key=(90,))
    mat = q4.Q4Matrix(to_dev(layer.qweight), to_dev(layer.qzeros), to_dev(layer.scales), None, to_dev(layer.bias), gs)
    check_layer_still_works(q4, mat, layer, K, N, gs)
    mat.close()


def test_allocation_failure_is_out_of_memory_and_recoverable(q4):
    K, N, gs = 1024, 256, 128
    layer = synthetic.make_layer(K, N, gs, act_order=True, bias=True, key=(92,))
    mat = q4.Q4Matrix(to_dev(layer.qweight), to_dev(layer.qzeros), to_dev(layer.scales), to_dev(layer.g_idx),
                      to_dev(layer.bias), gs)
    # temp_state for 2e8 rows of 1024 fp16 values is ~410 GB, past any GB300's memory
    with pytest.raises(q4.GPTQ4Error) as e:
        mat.reserve(200_000_000)
    assert e.value.status == q4.GPTQ_Q4_OUT_OF_MEMORY
    assert "temp_state" in e.value.message or "workspace" in e.value.message or "tickets" in e.value.message
    check_layer_still_works(q4, mat, layer, K, N, gs)
    mat.close()
