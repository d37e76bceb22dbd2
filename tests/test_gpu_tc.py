"""GPU parity of the tensor-core (tcgen05) paths: the dense fp16 GEMM on a
dequantized matrix, the unfused prefill (dequantize to temp_dq + GEMM) and
the fused prefill (shared-memory dequantization inside the GEMM main loop),
each against the CPU oracle, through the C ABI."""
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


def check(y_gpu, y_ref, tol, what):
    y = y_gpu.float().cpu().numpy().astype(np.float64)
    err = np.abs(y - y_ref)
    bad = err > tol
    ratio = float(np.max(err / np.maximum(tol, 1e-300)))
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside tolerance, worst err/tol {ratio:.3f}"
    return ratio


@pytest.mark.parametrize("M,K,N", [(1, 64, 64), (64, 128, 256), (128, 256, 320), (200, 1024, 512),
                                   (300, 576, 768), (513, 2048, 1024)])
def test_gemm_f16_matches_oracle(q4, M, K, N):
    g = np.random.default_rng(31 + M + K + N)
    a = g.standard_normal((M, K)).astype(np.float16)
    b = (g.standard_normal((K, N)) * 0.05).astype(np.float16)
    bias = (g.standard_normal(N) * 0.1).astype(np.float16)
    y = q4.gemm_f16(to_dev(a), to_dev(b), to_dev(bias))
    torch.cuda.synchronize()
    a64 = a.astype(np.float64)
    b64 = b.astype(np.float64)
    y_ref = oracle.linear_f64(a64, b64, bias.astype(np.float64))
    tol = oracle.tolerance(a, b, y_ref, K)
    check(y, y_ref, tol, f"gemm M={M} K={K} N={N}")


LAYERS = [  # (K, N, groupsize, act_order)
    (64, 64, 32, False),
    (256, 320, 64, False),
    (512, 256, 128, True),
    (1024, 448, 32, True),
    (1152, 576, 96, False),     # group of three 32-row blocks: some stages span two groups
    (2048, 512, -1, False),
    (1344, 320, 96, True),      # K split in two at stage 10: the second slice starts inside a group
]


@pytest.mark.parametrize("K,N,gs,act", LAYERS)
def test_prefill_fused_and_unfused_match_oracle(q4, K, N, gs, act):
    layer = synthetic.make_layer(K, N, gs, act_order=act, bias=True, key=(32, K, N, gs & 0xFFFF, act))
    dq = oracle.dequantize_layer(layer.qweight, layer.qzeros, layer.scales, layer.g_idx, K, N, gs)
    mat = q4.Q4Matrix(to_dev(layer.qweight), to_dev(layer.qzeros), to_dev(layer.scales), to_dev(layer.g_idx),
                      to_dev(layer.bias), gs)
    mat.set_path(q4.GPTQ_Q4_PATH_PREFILL)
    for M in (1, 5, 127, 128, 129, 300):
        x = synthetic.activations(M, K, key=(32, K, N, M))
        y_ref = oracle.reference_output(x, dq, layer.bias)
        tol = oracle.tolerance(x, dq.w16, y_ref, K)
        y = mat(to_dev(x))
        yu = mat.matmul_unfused(to_dev(x))
        torch.cuda.synchronize()
        check(y, y_ref, tol, f"fused K={K} N={N} g={gs} act={act} M={M}")
        check(yu, y_ref, tol, f"unfused K={K} N={N} g={gs} act={act} M={M}")
    mat.device_error()


@pytest.mark.parametrize("act", [False, True])
@pytest.mark.parametrize("K,N", synthetic.PREFILL_7B_SHAPES)
def test_prefill_7b_workload_sampled(q4, K, N, act):
    """Every prefill_7b case: the three Llama-7B shapes x {trivial, act-order}
    x M in {512, 2048}, full output on the GPU by the fused prefill, the
    unfused route and the decode path (past eight K slices: the last-arriver
    reduction), oracle on a row sample (all N columns of 24 seeded rows, plus
    the first and last row)."""
    layer = synthetic.workload_layer("prefill_7b", K, N, 128, act)
    dq = oracle.dequantize_layer(layer.qweight, layer.qzeros, layer.scales, layer.g_idx, K, N, 128)
    mat = q4.Q4Matrix(to_dev(layer.qweight), to_dev(layer.qzeros), to_dev(layer.scales), to_dev(layer.g_idx),
                      None, 128)
    for M in synthetic.PREFILL_7B_M:
        x = synthetic.workload_x("prefill_7b", K, N, 128, act, M)
        rows = np.unique(np.concatenate([[0, M - 1], np.random.default_rng(33 + M).choice(M, 24, replace=False)]))
        y_ref = oracle.reference_output(x[rows], dq)
        tol = oracle.tolerance(x, dq.w16, y_ref, K)
        xd = to_dev(x)
        mat.set_path(q4.GPTQ_Q4_PATH_AUTO)
        ya = mat(xd)
        mat.set_path(q4.GPTQ_Q4_PATH_PREFILL)
        y = mat(xd)
        yu = mat.matmul_unfused(xd)
        mat.set_path(q4.GPTQ_Q4_PATH_DECODE)
        yd = mat(xd)
        torch.cuda.synchronize()
        tr = torch.from_numpy(rows).to(DEV)
        what = f"{K}x{N} act={act} M={M}"
        check(ya[tr], y_ref, tol, f"default path {what}")
        check(y[tr], y_ref, tol, f"fused {what}")
        check(yu[tr], y_ref, tol, f"unfused {what}")
        check(yd[tr], y_ref, tol, f"decode path {what}")
        del ya, y, yu, yd
    mat.device_error()


@pytest.mark.parametrize("K,N,gs,act,M", [(1152, 576, 96, False, 4900), (1024, 448, 32, True, 7300),
                                          (1152, 576, 96, False, 9700), (1024, 448, 32, True, 14600)])
def test_prefill_wide_tiles_sampled(q4, K, N, gs, act, M):
    """Many rows on a narrow layer, with a ragged last column tile and a
    ragged last row tile: 256 x 256 tiles cut into two equal k ranges (the
    first two cases) or taken whole, round robin (the last two); oracle on a
    row sample."""
    layer = synthetic.make_layer(K, N, gs, act_order=act, bias=True, key=(34, K, N, gs & 0xFFFF, act))
    dq = oracle.dequantize_layer(layer.qweight, layer.qzeros, layer.scales, layer.g_idx, K, N, gs)
    mat = q4.Q4Matrix(to_dev(layer.qweight), to_dev(layer.qzeros), to_dev(layer.scales), to_dev(layer.g_idx),
                      to_dev(layer.bias), gs)
    x = synthetic.activations(M, K, key=(34, K, N, M))
    rows = np.unique(np.concatenate([[0, M - 1], np.random.default_rng(35).choice(M, 48, replace=False)]))
    y_ref = oracle.reference_output(x[rows], dq, layer.bias)
    tol = oracle.tolerance(x, dq.w16, y_ref, K)
    mat.set_path(q4.GPTQ_Q4_PATH_PREFILL)
    y = mat(to_dev(x))
    torch.cuda.synchronize()
    check(y[rows], y_ref, tol, f"fused wide tiles K={K} N={N} g={gs} act={act} M={M}")
    mat.device_error()


def test_prefill_stream_k_finish_matches_oracle(q4):
    """Stream-K ranges with tiles cut into two or three pieces, finished by
    the CTA holding each tile's piece 0 (from tensor memory, the other pieces
    staged into its ring memory): 80 column tiles of 256 on the GPU's SMs
    (fewer than two SMs per tile), a ragged last tile, bias, act-order, and
    fp16, bf16 (rows outside fp16's range) and fp32 activations, at 128- and
    256-row tiles."""
    K, N, gs = 1024, 20416, 128
    layer = synthetic.make_layer(K, N, gs, act_order=True, bias=True, key=(41, K, N))
    dq = oracle.dequantize_layer(layer.qweight, layer.qzeros, layer.scales, layer.g_idx, K, N, gs)
    mat = q4.Q4Matrix(to_dev(layer.qweight), to_dev(layer.qzeros), to_dev(layer.scales), to_dev(layer.g_idx),
                      to_dev(layer.bias), gs)
    mat.set_path(q4.GPTQ_Q4_PATH_PREFILL)
    scales = [1.0, 1e6, 1e-6, 3e4]
    for M in (40, 200, 300):
        x = synthetic.activations(M, K, key=(41, M))
        y_ref = oracle.reference_output(x, dq, layer.bias)
        y = mat(to_dev(x))
        torch.cuda.synchronize()
        check(y, y_ref, oracle.tolerance(x, dq.w16, y_ref, K), f"fp16 M={M}")
        rs = [scales[m % 4] for m in range(M)]
        mat.set_act_dtype(torch.bfloat16)
        xb = synthetic.activations_bf16(M, K, key=(42, M), row_scales=rs)
        yb = mat(torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).to(DEV).view(torch.bfloat16))
        torch.cuda.synchronize()
        yb_ref = oracle.reference_output_bf16(xb, dq, layer.bias)
        check(yb, yb_ref, oracle.tolerance_rows_bf16(xb, dq.w16, yb_ref, K), f"bf16 M={M}")
        mat.set_act_dtype(torch.float32)
        xf = synthetic.activations_f32(M, K, key=(43, M), row_scales=rs)
        yf = mat(torch.from_numpy(np.ascontiguousarray(xf).view(np.float32)).to(DEV))
        torch.cuda.synchronize()
        yf_ref = oracle.reference_output_f32(xf, dq, layer.bias)
        check(yf, yf_ref, oracle.tolerance_rows_f32(xf, dq.w16, yf_ref, K), f"fp32 M={M}")
        mat.set_act_dtype(torch.float16)
    mat.device_error()
