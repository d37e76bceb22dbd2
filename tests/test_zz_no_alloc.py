"""gptq_q4_matmul_noalloc: the decode matmul for callers that cannot allocate
device memory while they run a layer (a plugin in a framework that owns all
device memory, a service whose memory is budgeted up front, a loop that must
not hit cudaMalloc's device-wide synchronization).  Its scratch lives in one
fixed device array inside the library.

Checked through the C ABI, on two calls in a row, element by element against
the CPU oracle within the tolerance the other parity tests use, and against
the ordinary entry point, gptq_q4_matmul, within the same tolerance.
Collected last (file name) so that a run stopping at its first failure has
already run every other test."""
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


@pytest.mark.parametrize("K,N,gs,act,M", [
    (4096, 4096, 128, False, 1),      # K slices reduced inside a thread-block cluster
    (28672, 1024, 128, False, 16),    # 14 K slices: partial sums and tickets in the scratch
    (4096, 11008, 128, True, 4),      # act-order: temp_state in the scratch
    (11008, 4096, 128, False, 8),
    (1024, 448, 32, True, 17),        # two m-tiles, ragged rows
])
def test_noalloc_matches_matmul_two_calls_in_a_row(q4, K, N, gs, act, M):
    layer = synthetic.make_layer(K, N, gs, act_order=act, bias=True, key=(41, K, N, gs, act))
    dq = oracle.dequantize_layer(layer.qweight, layer.qzeros, layer.scales, layer.g_idx, K, N, gs)
    mat = q4.Q4Matrix(to_dev(layer.qweight), to_dev(layer.qzeros), to_dev(layer.scales), to_dev(layer.g_idx),
                      to_dev(layer.bias), gs)
    mat.set_path(q4.GPTQ_Q4_PATH_DECODE)
    x = synthetic.activations(M, K, key=(41, K, N, M))
    xd = to_dev(x)
    stream = torch.cuda.current_stream().cuda_stream
    ref = torch.empty((M, N), dtype=torch.float16, device=DEV)
    q4.gptq_q4_matmul(mat.handle, xd.data_ptr(), M, ref.data_ptr(), stream)
    y_oracle = oracle.reference_output(x, dq, layer.bias)
    tol = oracle.tolerance(x, dq.w16, y_oracle, K)
    bytes_before = mat.info()["device_bytes"]
    for call in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
        q4.gptq_q4_matmul_noalloc(mat.handle, xd.data_ptr(), M, out.data_ptr(), stream)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy().astype(np.float64)
        err = np.abs(got - y_oracle)
        assert np.all(err <= tol), f"call {call}: worst |noalloc - oracle| / tol {float(np.max(err / tol)):.3f}"
        diff = np.abs(got - ref.float().cpu().numpy().astype(np.float64))
        assert np.all(diff <= tol), f"call {call}: worst |noalloc - matmul| / tol {float(np.max(diff / tol)):.3f}"
    assert mat.info()["device_bytes"] == bytes_before
    mat.device_error()
    mat.close()


def test_noalloc_never_grows_the_handle(q4):
    """A row count past what the handle's own buffers were sized for: the
    ordinary call would grow them; this one uses the fixed scratch."""
    K, N, gs, M = 4096, 4096, 128, 48
    layer = synthetic.make_layer(K, N, gs, act_order=True, key=(42,))
    mat = q4.Q4Matrix(to_dev(layer.qweight), to_dev(layer.qzeros), to_dev(layer.scales), to_dev(layer.g_idx),
                      None, gs)
    before = mat.info()["device_bytes"]
    x = synthetic.activations(M, K, key=(42, M))
    out = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    q4.gptq_q4_matmul_noalloc(mat.handle, to_dev(x).data_ptr(), M, out.data_ptr(),
                              torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert mat.info()["device_bytes"] == before
    dq = oracle.dequantize_layer(layer.qweight, layer.qzeros, layer.scales, layer.g_idx, K, N, gs)
    y_oracle = oracle.reference_output(x, dq)
    tol = oracle.tolerance(x, dq.w16, y_oracle, K)
    err = np.abs(out.float().cpu().numpy().astype(np.float64) - y_oracle)
    assert np.all(err <= tol), f"worst |noalloc - oracle| / tol {float(np.max(err / tol)):.3f}"
    mat.device_error()
    mat.close()


def test_noalloc_rejects_sizes_beyond_the_scratch(q4):
    K, N, gs = 8192, 28672, 128
    layer = synthetic.make_layer(K, N, gs, act_order=True, key=(43,))
    mat = q4.Q4Matrix(to_dev(layer.qweight), to_dev(layer.qzeros), to_dev(layer.scales), to_dev(layer.g_idx),
                      None, gs)
    M = 2048                                 # act-order temp_state alone: 2048 x 8192 x 2 B = 32 MiB
    x = torch.zeros((M, K), dtype=torch.float16, device=DEV)
    out = torch.empty((M, N), dtype=torch.float16, device=DEV)
    with pytest.raises(q4.GPTQ4Error) as e:
        q4.gptq_q4_matmul_noalloc(mat.handle, x.data_ptr(), M, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert e.value.status == q4.GPTQ_Q4_INVALID_ARGUMENT
    assert str(q4.GPTQ_Q4_NOALLOC_SCRATCH_BYTES) in e.value.message
    mat.close()
