"""GPU parity of the C-ABI path against the CPU oracle.

Codes and dequantized weights must match bit for bit; y must be within
1e-2 sqrt(K) max|x| max|w| / 64 + 2e-3 |y_ref| per element.  Every call goes
through the C ABI (via the ctypes binding); inputs are seeded and synthetic.
"""
import numpy as np
import pytest

import oracle
import synthetic

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gptq_bit_weight_gb300 as q4mod
    return q4mod


DEV = "cuda:0"


def to_dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def make(q4, layer, bias=True):
    return q4.Q4Matrix(to_dev(layer.qweight), to_dev(layer.qzeros), to_dev(layer.scales), to_dev(layer.g_idx),
                       to_dev(layer.bias) if bias else None, layer.groupsize)


def oracle_dq(layer):
    return oracle.dequantize_layer(layer.qweight, layer.qzeros, layer.scales, layer.g_idx, layer.K, layer.N,
                                   layer.groupsize)


def check_y(y_gpu, x, dq, bias, K, what=""):
    y_ref = oracle.reference_output(x, dq, bias)
    tol = oracle.tolerance(x, dq.w16, y_ref, K)
    y = y_gpu.float().cpu().numpy().astype(np.float64)
    err = np.abs(y - y_ref)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements outside tolerance; worst err/tol "
                           f"{float(np.max(err / np.maximum(tol, 1e-300))):.3f}")
    return float(np.max(err / np.maximum(tol, 1e-300)))


SMALL = [  # (K, N, groupsize, act_order)
    (64, 64, 32, False),
    (256, 128, 64, False),
    (256, 192, -1, False),
    (512, 320, 128, True),
    (1024, 448, 32, True),
    (1088, 576, 64, False),     # K not a multiple of the split slices -> ragged chunks
    (1152, 320, 96, True),      # group of three 32-row blocks
    (2048, 960, 128, False),
    (1024, 256, -1, True),      # one group: act-order reduces to the identity
]


@pytest.mark.parametrize("K,N,gs,act", SMALL)
def test_unpack_and_dequant_bit_exact(q4, K, N, gs, act):
    layer = synthetic.make_layer(K, N, gs, act_order=act, key=(21, K, N, gs & 0xFFFF, act))
    dq = oracle_dq(layer)
    mat = make(q4, layer, bias=False)
    q, z = mat.debug_unpack()
    w = mat.dequant()
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), dq.q)
    assert np.array_equal(z.cpu().numpy(), dq.z)
    assert np.array_equal(w.cpu().numpy().view(np.uint16), dq.w16)
    mat.device_error()


@pytest.mark.parametrize("path", ["DECODE", "DECODE_RING", "DECODE_MMA", "DECODE_TC", "DECODE_STREAM"])
@pytest.mark.parametrize("K,N,gs,act", SMALL)
def test_decode_matches_oracle(q4, K, N, gs, act, path):
    """Every decode kernel: DECODE_RING runs the TMA-ring kernel for M <= 16
    (register-streaming above); DECODE_MMA always the register-streaming one;
    DECODE_TC the tcgen05 one with per-group accumulators for M <= 16; DECODE
    chooses by layer size and M (on these small layers: register-streaming)."""
    layer = synthetic.make_layer(K, N, gs, act_order=act, bias=True, key=(22, K, N, gs & 0xFFFF, act))
    dq = oracle_dq(layer)
    mat = make(q4, layer)
    mat.set_path(getattr(q4, "GPTQ_Q4_PATH_" + path))
    for M in (1, 2, 3, 4, 7, 8, 9, 16, 17, 33, 40):
        x = synthetic.activations(M, K, key=(22, K, N, M))
        y = mat(to_dev(x))
        torch.cuda.synchronize()
        check_y(y, x, dq, layer.bias, K, f"{path} K={K} N={N} g={gs} act={act} M={M}")
    mat.device_error()


RING_SLOT_CASES = [  # (K, N, groupsize, act_order)
    (4096, 256, 32, False),     # 16 groups per slice: two full batches of 8 group slots at M = 1
    (2304, 192, 96, True),      # 320-row slices start inside groups; a 64-column last tile idles two warps
    (1024, 128, -1, False),     # one group for the whole K
    (6144, 128, 64, True),      # many groups, few tiles: the widest K split
]


@pytest.mark.parametrize("K,N,gs,act", RING_SLOT_CASES)
def test_ring_group_slots_match_oracle(q4, K, N, gs, act):
    """TMA-ring decode with M <= 4: spare MMA columns carry consecutive
    quantization groups (a batch of 8 / MP groups per flush, MP = M rounded up
    to a power of two), summed across lanes at the end; M = 5 and 8 run
    without slots."""
    layer = synthetic.make_layer(K, N, gs, act_order=act, bias=True, key=(27, K, N, gs & 0xFFFF, act))
    dq = oracle_dq(layer)
    mat = make(q4, layer)
    mat.set_path(q4.GPTQ_Q4_PATH_DECODE_RING)
    for M in (1, 2, 3, 4, 5, 8):
        x = synthetic.activations(M, K, key=(27, K, N, M))
        y = mat(to_dev(x))
        torch.cuda.synchronize()
        check_y(y, x, dq, layer.bias, K, f"ring slots K={K} N={N} g={gs} act={act} M={M}")
    mat.device_error()


UNEVEN_CASES = [  # (K, N, groupsize, empty group)
    (1024, 256, 128, None),
    (2048, 320, 64, None),
    (1024, 192, 256, 2),        # one group holds no row at all
]


@pytest.mark.parametrize("K,N,gs,empty", UNEVEN_CASES)
def test_uneven_groups_match_oracle(q4, K, N, gs, empty):
    """g_idx with groups of unequal size: the handle pads every group to the
    largest one (whole 32-row blocks) with zero-x rows; codes, dequantized
    weights and y on every path against the oracle, which takes any g_idx."""
    import dataclasses
    base = synthetic.make_layer(K, N, gs, bias=True, key=(29, K, N, gs))
    gi = synthetic.uneven_group_index(K, K // gs, key=(29, K, gs), empty_group=empty)
    assert len(set(np.bincount(gi, minlength=K // gs).tolist())) > 1
    layer = dataclasses.replace(base, g_idx=gi, act_order=True)
    dq = oracle_dq(layer)
    mat = make(q4, layer)
    info = mat.info()
    assert info["K"] == K and info["act_order"]
    q, z = mat.debug_unpack()
    w = mat.dequant()
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), dq.q)
    assert np.array_equal(z.cpu().numpy(), dq.z)
    assert np.array_equal(w.cpu().numpy().view(np.uint16), dq.w16)
    for path in ("AUTO", "DECODE", "DECODE_RING", "DECODE_MMA", "DECODE_STREAM", "PREFILL"):
        mat.set_path(getattr(q4, "GPTQ_Q4_PATH_" + path))
        for M in (1, 5, 33, 300):
            x = synthetic.activations(M, K, key=(29, K, N, M))
            y = mat(to_dev(x))
            torch.cuda.synchronize()
            check_y(y, x, dq, layer.bias, K, f"uneven {path} K={K} N={N} g={gs} M={M}")
    x = synthetic.activations(40, K, key=(29, K, N, 40))
    yu = mat.matmul_unfused(to_dev(x))
    torch.cuda.synchronize()
    check_y(yu, x, dq, layer.bias, K, f"uneven unfused K={K} N={N} g={gs}")
    mat.device_error()


@pytest.mark.parametrize("act", [False, True])
def test_groupsize_not_multiple_of_32(q4, act):
    """groupsize 48: each group is padded to 64 rows inside the handle, with
    or without act-order; every path against the oracle."""
    K, N, gs = 960, 192, 48
    layer = synthetic.make_layer(K, N, gs, act_order=act, bias=True, key=(30, K, N, gs, act))
    dq = oracle_dq(layer)
    mat = make(q4, layer)
    assert mat.info()["K"] == K
    w = mat.dequant()
    torch.cuda.synchronize()
    assert np.array_equal(w.cpu().numpy().view(np.uint16), dq.w16)
    for path in ("AUTO", "DECODE", "DECODE_RING", "DECODE_MMA", "DECODE_STREAM", "PREFILL"):
        mat.set_path(getattr(q4, "GPTQ_Q4_PATH_" + path))
        for M in (1, 6, 40):
            x = synthetic.activations(M, K, key=(30, K, N, M))
            y = mat(to_dev(x))
            torch.cuda.synchronize()
            check_y(y, x, dq, layer.bias, K, f"g=48 {path} act={act} M={M}")
    mat.device_error()


EIGHT_BIT_CASES = [  # (K, N, groupsize, act_order)
    (256, 128, 64, False),
    (1024, 448, 32, True),
    (1152, 320, 96, True),
    (1024, 256, -1, False),
    (2048, 960, 128, False),
]


@pytest.mark.parametrize("K,N,gs,act", EIGHT_BIT_CASES)
def test_8bit_matches_oracle(q4, K, N, gs, act):
    """8-bit checkpoints (qweight [K/4][N], qzeros [G][N/4]) held as two 4-bit
    halves: the codes, zero points and dequantized weights bit for bit, y on
    every path, GPTQ and GPTQ_V2 zero conventions."""
    layer = synthetic.make_layer8(K, N, gs, act_order=act, bias=True, key=(31, K, N, gs & 0xFFFF, act))
    mat = q4.Q4Matrix(to_dev(layer.qweight), to_dev(layer.qzeros), to_dev(layer.scales), to_dev(layer.g_idx),
                      to_dev(layer.bias), gs, bits=8)
    info = mat.info()
    assert info["K"] == K and info["G"] == layer.G
    for fmt, zo in ((q4.GPTQ_Q4_FORMAT_GPTQ, 1), (q4.GPTQ_Q4_FORMAT_GPTQ_V2, 0)):
        mat.set_format(fmt)
        dq = oracle.dequantize_layer(layer.qweight, layer.qzeros, layer.scales, layer.g_idx, K, N, gs,
                                     zero_offset=zo, bits=8)
        q, z = mat.debug_unpack()
        w = mat.dequant()
        torch.cuda.synchronize()
        assert np.array_equal(q.cpu().numpy(), dq.q)
        assert np.array_equal(z.cpu().numpy(), dq.z)
        assert np.array_equal(w.cpu().numpy().view(np.uint16), dq.w16)
        for path in ("AUTO", "DECODE", "DECODE_RING", "DECODE_MMA", "DECODE_TC", "DECODE_STREAM", "PREFILL"):
            mat.set_path(getattr(q4, "GPTQ_Q4_PATH_" + path))
            for M in (1, 3, 8, 16, 40):
                x = synthetic.activations(M, K, key=(31, K, N, M))
                y = mat(to_dev(x))
                torch.cuda.synchronize()
                check_y(y, x, dq, layer.bias, K, f"8-bit {path} fmt={fmt} K={K} N={N} g={gs} act={act} M={M}")
        x = synthetic.activations(300, K, key=(31, K, N, 300))
        mat.set_path(q4.GPTQ_Q4_PATH_AUTO)
        y = mat(to_dev(x))
        yu = mat.matmul_unfused(to_dev(x))
        torch.cuda.synchronize()
        check_y(y, x, dq, layer.bias, K, f"8-bit prefill fmt={fmt} M=300")
        check_y(yu, x, dq, layer.bias, K, f"8-bit unfused fmt={fmt} M=300")
    mat.device_error()
    mat.close()


def test_8bit_llama7b_shape(q4):
    """An 8-bit 4096 x 11008 layer (g = 128): decode at M = 1 and 8 and the
    fused prefill at M = 512 (oracle on a row sample)."""
    K, N, gs = 4096, 11008, 128
    layer = synthetic.make_layer8(K, N, gs, bias=True, key=(32, K, N))
    dq = oracle.dequantize_layer(layer.qweight, layer.qzeros, layer.scales, None, K, N, gs, bits=8)
    mat = q4.Q4Matrix(to_dev(layer.qweight), to_dev(layer.qzeros), to_dev(layer.scales), None,
                      to_dev(layer.bias), gs, bits=8)
    w = mat.dequant()
    torch.cuda.synchronize()
    assert np.array_equal(w.cpu().numpy().view(np.uint16), dq.w16)
    del w
    for M in (1, 8):
        x = synthetic.activations(M, K, key=(32, K, N, M))
        y = mat(to_dev(x))
        torch.cuda.synchronize()
        check_y(y, x, dq, layer.bias, K, f"8-bit 7B M={M}")
    M = 512
    x = synthetic.activations(M, K, key=(32, K, N, M))
    rows = np.unique(np.concatenate([[0, M - 1], np.random.default_rng(36).choice(M, 16, replace=False)]))
    y = mat(to_dev(x))
    torch.cuda.synchronize()
    check_y(y[rows], x[rows], dq, layer.bias, K, "8-bit 7B M=512")
    mat.device_error()
    mat.close()


BF16_CASES = [  # (K, N, groupsize, act_order)
    (256, 128, 64, False),
    (1024, 448, 32, True),
    (1152, 320, 96, True),
    (2048, 960, 128, False),
]
BF16_ROW_SCALES = [1.0, 1e6, 1e-6, 3e4]     # rows beyond fp16's range both ways


def bf16_tensor(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def check_y_bf16(y_gpu, xb, dq, bias, K, what=""):
    y_ref = oracle.reference_output_bf16(xb, dq, bias)
    tol = oracle.tolerance_rows_bf16(xb, dq.w16, y_ref, K)
    y = y_gpu.float().cpu().numpy().astype(np.float64)
    err = np.abs(y - y_ref)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements outside tolerance; worst err/tol "
                           f"{float(np.max(err / np.maximum(tol, 1e-300))):.3f}")


@pytest.mark.parametrize("K,N,gs,act", BF16_CASES)
def test_bf16_activations_match_oracle(q4, K, N, gs, act):
    """bf16 x and y: every path (and the unfused route and the
    allocation-free call) against the oracle, with rows of x scaled by 1e6 and
    1e-6 (outside fp16's range), checked row by row."""
    layer = synthetic.make_layer(K, N, gs, act_order=act, bias=True, key=(33, K, N, gs & 0xFFFF, act))
    dq = oracle_dq(layer)
    mat = make(q4, layer)
    mat.set_act_dtype(torch.bfloat16)
    for path in ("AUTO", "DECODE", "DECODE_RING", "DECODE_MMA", "DECODE_TC", "DECODE_STREAM", "PREFILL"):
        mat.set_path(getattr(q4, "GPTQ_Q4_PATH_" + path))
        for M in (1, 3, 8, 16, 40):
            rs = [BF16_ROW_SCALES[m % 4] for m in range(M)]
            xb = synthetic.activations_bf16(M, K, key=(33, K, N, M), row_scales=rs)
            y = mat(bf16_tensor(xb))
            torch.cuda.synchronize()
            assert y.dtype == torch.bfloat16
            check_y_bf16(y, xb, dq, layer.bias, K, f"bf16 {path} K={K} N={N} g={gs} act={act} M={M}")
    M = 300
    xb = synthetic.activations_bf16(M, K, key=(33, K, N, M), row_scales=[BF16_ROW_SCALES[m % 4] for m in range(M)])
    mat.set_path(q4.GPTQ_Q4_PATH_AUTO)
    y = mat(bf16_tensor(xb))
    yu = mat.matmul_unfused(bf16_tensor(xb))
    torch.cuda.synchronize()
    check_y_bf16(y, xb, dq, layer.bias, K, "bf16 prefill M=300")
    check_y_bf16(yu, xb, dq, layer.bias, K, "bf16 unfused M=300")
    M = 4
    xb = synthetic.activations_bf16(M, K, key=(34, K, N, M), row_scales=BF16_ROW_SCALES)
    xt = bf16_tensor(xb)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    q4.gptq_q4_matmul_noalloc(mat.handle, xt.data_ptr(), M, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    check_y_bf16(out, xb, dq, layer.bias, K, "bf16 noalloc M=4")
    mat.set_act_dtype(torch.float16)
    x = synthetic.activations(5, K, key=(33, K, N, 5))
    y = mat(to_dev(x))
    torch.cuda.synchronize()
    check_y(y, x, dq, layer.bias, K, "back to fp16")
    mat.device_error()


def f32_tensor(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.float32)).to(DEV)


def check_y_f32(y_gpu, xf, dq, bias, K, what=""):
    y_ref = oracle.reference_output_f32(xf, dq, bias)
    tol = oracle.tolerance_rows_f32(xf, dq.w16, y_ref, K)
    y = y_gpu.cpu().numpy().astype(np.float64)
    err = np.abs(y - y_ref)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements outside tolerance; worst err/tol "
                           f"{float(np.max(err / np.maximum(tol, 1e-300))):.3f}")


@pytest.mark.parametrize("K,N,gs,act", BF16_CASES)
def test_f32_activations_match_oracle(q4, K, N, gs, act):
    """fp32 x and y: every path and the unfused route against the oracle,
    with rows of x scaled by 1e6 and 1e-6 (outside fp16's range), checked
    row by row; the allocation-free call refuses an fp32 handle."""
    layer = synthetic.make_layer(K, N, gs, act_order=act, bias=True, key=(36, K, N, gs & 0xFFFF, act))
    dq = oracle_dq(layer)
    mat = make(q4, layer)
    mat.set_act_dtype(torch.float32)
    for path in ("AUTO", "DECODE", "DECODE_RING", "DECODE_MMA", "DECODE_TC", "DECODE_STREAM", "PREFILL"):
        mat.set_path(getattr(q4, "GPTQ_Q4_PATH_" + path))
        for M in (1, 3, 8, 16, 40):
            rs = [BF16_ROW_SCALES[m % 4] for m in range(M)]
            xf = synthetic.activations_f32(M, K, key=(36, K, N, M), row_scales=rs)
            y = mat(f32_tensor(xf))
            torch.cuda.synchronize()
            assert y.dtype == torch.float32
            check_y_f32(y, xf, dq, layer.bias, K, f"fp32 {path} K={K} N={N} g={gs} act={act} M={M}")
    M = 300
    xf = synthetic.activations_f32(M, K, key=(36, K, N, M), row_scales=[BF16_ROW_SCALES[m % 4] for m in range(M)])
    mat.set_path(q4.GPTQ_Q4_PATH_AUTO)
    y = mat(f32_tensor(xf))
    yu = mat.matmul_unfused(f32_tensor(xf))
    torch.cuda.synchronize()
    check_y_f32(y, xf, dq, layer.bias, K, "fp32 prefill M=300")
    check_y_f32(yu, xf, dq, layer.bias, K, "fp32 unfused M=300")
    out = torch.empty((4, N), dtype=torch.float32, device=DEV)
    xt = f32_tensor(synthetic.activations_f32(4, K, key=(37, K, N, 4)))
    with pytest.raises(q4.GPTQ4Error) as e:
        q4.gptq_q4_matmul_noalloc(mat.handle, xt.data_ptr(), 4, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert e.value.status == q4.GPTQ_Q4_UNSUPPORTED
    mat.set_act_dtype(torch.float16)
    x = synthetic.activations(5, K, key=(36, K, N, 5))
    y = mat(to_dev(x))
    torch.cuda.synchronize()
    check_y(y, x, dq, layer.bias, K, "back to fp16")
    mat.device_error()


def test_f32_activations_70b_shape(q4):
    """fp32 activations on a Llama-70B projection (8192 x 10240, act-order,
    g = 128) at decode and prefill sizes; oracle on a column sample."""
    K, N, gs = 8192, 10240, 128
    layer = synthetic.workload_layer("sweep_70b", K, N, gs, True)
    g = np.random.default_rng(38)
    blocks = np.sort(g.choice(N // 8, size=16, replace=False))
    cols = (blocks[:, None] * 8 + np.arange(8)[None, :]).reshape(-1)
    dq = oracle.dequantize_layer(layer.qweight[:, cols], layer.qzeros[:, blocks], layer.scales[:, cols],
                                 layer.g_idx, K, cols.size, gs)
    mat = q4.Q4Matrix(to_dev(layer.qweight), to_dev(layer.qzeros), to_dev(layer.scales), to_dev(layer.g_idx),
                      None, gs)
    mat.set_act_dtype(torch.float32)
    tcols = torch.from_numpy(cols).to(DEV)
    for M in (1, 4, 64):
        xf = synthetic.activations_f32(M, K, key=(38, M), row_scales=[BF16_ROW_SCALES[m % 4] for m in range(M)])
        y = mat(f32_tensor(xf))
        torch.cuda.synchronize()
        check_y_f32(y[:, tcols], xf, dq, None, K, f"fp32 70B M={M}")
    mat.device_error()


V2_CASES = [  # (K, N, groupsize, act_order)
    (256, 128, 64, False),
    (1024, 448, 32, True),
    (1152, 320, 96, True),
    (2048, 960, 128, False),
]


@pytest.mark.parametrize("K,N,gs,act", V2_CASES)
def test_gptq_v2_format_matches_oracle(q4, K, N, gs, act):
    """GPTQ_V2 checkpoints (effective zero = stored zero): dequant bit for bit,
    every decode kernel and the fused prefill within tolerance, against the
    oracle run with the same convention; stored zeros include 0, whose
    effective zero lies below every GPTQ one."""
    layer = synthetic.make_layer(K, N, gs, act_order=act, bias=True, key=(25, K, N, gs & 0xFFFF, act))
    dq = oracle.dequantize_layer(layer.qweight, layer.qzeros, layer.scales, layer.g_idx, K, N, gs, zero_offset=0)
    assert np.any(dq.z == 0)
    mat = make(q4, layer)
    mat.set_format(q4.GPTQ_Q4_FORMAT_GPTQ_V2)
    w = mat.dequant()
    torch.cuda.synchronize()
    assert np.array_equal(w.cpu().numpy().view(np.uint16), dq.w16)
    for path in ("DECODE", "DECODE_RING", "DECODE_MMA", "DECODE_TC", "DECODE_STREAM", "PREFILL"):
        mat.set_path(getattr(q4, "GPTQ_Q4_PATH_" + path))
        for M in (1, 3, 8, 16, 40):
            x = synthetic.activations(M, K, key=(25, K, N, M))
            y = mat(to_dev(x))
            yu = mat.matmul_unfused(to_dev(x)) if path == "PREFILL" else None
            torch.cuda.synchronize()
            check_y(y, x, dq, layer.bias, K, f"v2 {path} K={K} N={N} g={gs} act={act} M={M}")
            if yu is not None:
                check_y(yu, x, dq, layer.bias, K, f"v2 unfused K={K} N={N} g={gs} act={act} M={M}")
    mat.set_format(q4.GPTQ_Q4_FORMAT_GPTQ)
    dq1 = oracle_dq(layer)
    mat.set_path(q4.GPTQ_Q4_PATH_AUTO)
    x = synthetic.activations(4, K, key=(25, K, N, 4))
    y = mat(to_dev(x))
    torch.cuda.synchronize()
    check_y(y, x, dq1, layer.bias, K, "back to GPTQ")
    with pytest.raises(q4.GPTQ4Error):
        mat.set_format(7)
    mat.device_error()


def test_trivial_gidx_same_as_none(q4):
    K, N, gs = 512, 256, 64
    layer = synthetic.make_layer(K, N, gs, key=(23,))
    x = to_dev(synthetic.activations(5, K, key=(23, 5)))
    a = make(q4, layer, bias=False)
    gi = to_dev((np.arange(K) // gs).astype(np.int32))
    b = q4.Q4Matrix(to_dev(layer.qweight), to_dev(layer.qzeros), to_dev(layer.scales), gi, None, gs)
    assert b.info()["act_order"] is False
    ya, yb = a(x), b(x)
    torch.cuda.synchronize()
    assert torch.equal(ya, yb)


@pytest.mark.parametrize("path", ["AUTO", "DECODE_STREAM", "DECODE_MMA", "PREFILL"])
def test_deterministic_repeat(q4, path):
    """Split reductions sum in a fixed order (slices, segments or pieces),
    never in arrival order: repeated calls give identical bits.  28672 rows
    cut the stream-K decode's tiles into several segments and the fused
    prefill's into several pieces."""
    K, N, gs = 28672, 1024, 128
    layer = synthetic.make_layer(K, N, gs, act_order=True, bias=True, key=(24,))
    mat = make(q4, layer)
    mat.set_path(getattr(q4, "GPTQ_Q4_PATH_" + path))
    for M in (1, 4, 300):
        x = to_dev(synthetic.activations(M, K, key=(24, M)))
        y1 = mat(x).clone()
        y2 = mat(x).clone()
        torch.cuda.synchronize()
        assert torch.equal(y1, y2), f"{path} M={M}"


def test_zero_rows_is_noop(q4):
    layer = synthetic.make_layer(256, 128, 64, key=(25,))
    mat = make(q4, layer, bias=False)
    x = torch.empty((0, 256), dtype=torch.float16, device=DEV)
    y = mat(x)
    assert y.shape == (0, 128)


def test_no_dense_weight_cache(q4):
    """The handle keeps the packed bytes plus O(G N + K) metadata, never K*N*2."""
    K, N, gs = 4096, 4096, 128
    layer = synthetic.make_layer(K, N, gs, act_order=True, key=(26,))
    mat = make(q4, layer, bias=False)
    info = mat.info()
    packed = K * N // 2
    meta = layer.G * N * 4 + layer.G * N // 2 + K * 4
    split_k = 16 * N * 4 * 8   # split-K partials for up to 16 rows, at most 8 slices
    assert info["device_bytes"] <= packed + meta + split_k + 4096
    assert info["device_bytes"] < K * N * 2 // 2


# ----------------------------------------------------------- workloads

def test_single_layer_workload(q4):
    layer, x = synthetic.single_layer()
    dq = oracle_dq(layer)
    mat = make(q4, layer, bias=False)
    y = mat(to_dev(x))
    torch.cuda.synchronize()
    check_y(y, x, dq, None, layer.K, "single_layer")


@pytest.mark.parametrize("K,N", synthetic.DECODE_7B_SHAPES)
def test_decode_7b_workload(q4, K, N):
    layer = synthetic.workload_layer("decode_7b", K, N, 128, False)
    dq = oracle_dq(layer)
    mat = make(q4, layer)
    q, z = mat.debug_unpack()
    w = mat.dequant()
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), dq.q)
    assert np.array_equal(w.cpu().numpy().view(np.uint16), dq.w16)
    for M in synthetic.DECODE_7B_M:
        x = synthetic.workload_x("decode_7b", K, N, 128, False, M)
        y = mat(to_dev(x))
        torch.cuda.synchronize()
        check_y(y, x, dq, layer.bias, K, f"decode_7b {K}x{N} M={M}")
    # the register-streaming kernel at every M <= 8 it serves: shared weight
    # ring with the x slice staged (short x slices) or carried per chunk
    # (long ones), and the raw-pair variant where its grid is one wave
    mat.set_path(q4.GPTQ_Q4_PATH_DECODE_MMA)
    for M in (1, 2, 3, 5, 8):
        x = synthetic.activations(M, K, key=(28, K, N, M))
        y = mat(to_dev(x))
        torch.cuda.synchronize()
        check_y(y, x, dq, layer.bias, K, f"register decode {K}x{N} M={M}")
    mat.device_error()


@pytest.mark.parametrize("K,N", synthetic.ACTORDER_7B_SHAPES)
def test_actorder_7b_workload(q4, K, N):
    layer = synthetic.workload_layer("actorder_7b", K, N, 128, True)
    dq = oracle_dq(layer)
    mat = make(q4, layer)
    assert mat.info()["act_order"]
    w = mat.dequant()
    torch.cuda.synchronize()
    assert np.array_equal(w.cpu().numpy().view(np.uint16), dq.w16)
    for M in synthetic.ACTORDER_7B_M:
        x = synthetic.workload_x("actorder_7b", K, N, 128, True, M)
        y = mat(to_dev(x))
        torch.cuda.synchronize()
        check_y(y, x, dq, None, K, f"actorder_7b {K}x{N} M={M}")


# --------------------------------------------------------- error codes

def test_error_codes(q4):
    from gptq_bit_weight_gb300 import GPTQ4Error
    qw = torch.zeros((32, 256), dtype=torch.int32, device=DEV)
    qz = torch.zeros((2, 32), dtype=torch.int32, device=DEV)
    sc = torch.ones((2, 256), dtype=torch.float16, device=DEV)
    with pytest.raises(GPTQ4Error) as e:
        q4.gptq_q4_make(qw.data_ptr(), qz.data_ptr(), sc.data_ptr(), None, 256, 256, 100)
    assert e.value.status == q4.GPTQ_Q4_INVALID_ARGUMENT
    with pytest.raises(GPTQ4Error) as e:
        q4.gptq_q4_make(qw.data_ptr(), qz.data_ptr(), sc.data_ptr(), None, 256, 250, 128)
    assert e.value.status == q4.GPTQ_Q4_INVALID_ARGUMENT
    with pytest.raises(GPTQ4Error) as e:       # valid GPTQ, but the GPU layout needs N % 64
        q4.gptq_q4_make(qw.data_ptr(), qz.data_ptr(), sc.data_ptr(), None, 256, 200, 128)
    assert e.value.status in (q4.GPTQ_Q4_UNSUPPORTED, q4.GPTQ_Q4_INVALID_ARGUMENT)
    gi = torch.zeros(256, dtype=torch.int32, device=DEV)
    gi[3] = 2                                   # outside [0, G)
    with pytest.raises(GPTQ4Error) as e:
        q4.gptq_q4_make(qw.data_ptr(), qz.data_ptr(), sc.data_ptr(), gi.data_ptr(), 256, 256, 128)
    assert e.value.status == q4.GPTQ_Q4_INVALID_ARGUMENT
    gi = torch.zeros(256, dtype=torch.int32, device=DEV)   # eight groups of 32, all rows in the first:
    qz8 = torch.zeros((8, 32), dtype=torch.int32, device=DEV)
    sc8 = torch.ones((8, 256), dtype=torch.float16, device=DEV)
    with pytest.raises(GPTQ4Error) as e:       # padding every group to 256 rows would be 8x the checkpoint
        q4.gptq_q4_make(qw.data_ptr(), qz8.data_ptr(), sc8.data_ptr(), gi.data_ptr(), 256, 256, 32)
    assert e.value.status == q4.GPTQ_Q4_UNSUPPORTED
    host = np.zeros((32, 256), np.int32)
    with pytest.raises(GPTQ4Error) as e:       # host pointer
        q4.gptq_q4_make(host.ctypes.data, qz.data_ptr(), sc.data_ptr(), None, 256, 256, 128)
    assert e.value.status == q4.GPTQ_Q4_INVALID_ARGUMENT
    h = q4.gptq_q4_make(qw.data_ptr(), qz.data_ptr(), sc.data_ptr(), None, 256, 256, 128)
    try:
        x = torch.zeros((4, 256), dtype=torch.float16, device=DEV)
        out = torch.empty((4, 256), dtype=torch.float16, device=DEV)
        with pytest.raises(GPTQ4Error) as e:   # misaligned x
            q4.gptq_q4_matmul(h, x.data_ptr() + 2, 3, out.data_ptr(), 0)
        assert e.value.status == q4.GPTQ_Q4_INVALID_ARGUMENT
        with pytest.raises(GPTQ4Error) as e:
            q4.gptq_q4_matmul(h, x.data_ptr(), -1, out.data_ptr(), 0)
        assert e.value.status == q4.GPTQ_Q4_INVALID_ARGUMENT
        assert q4.gptq_q4_matmul(h, 0, 0, 0, 0) == 0
    finally:
        q4.gptq_q4_free(h)


@pytest.mark.parametrize("act", [False, True])
def test_fused_projections_match_oracle(q4, act):
    """Three projections of one input (widths 256, 128, 320) in one handle:
    dequant bit for bit and every path within tolerance against the oracle of
    the N-concatenated checkpoint; each part's columns against that part's own
    oracle."""
    K, gs, Ns = 1024, 128, [256, 128, 320]
    base = synthetic.make_layer(K, sum(Ns), gs, act_order=act, bias=True, key=(26, K, act))
    parts, off = [], 0
    for n in Ns:
        parts.append((base.qweight[:, off:off + n], base.qzeros[:, off // 8:(off + n) // 8],
                      base.scales[:, off:off + n], base.bias[off:off + n]))
        off += n
    mat = q4.Q4Matrix.fused([(to_dev(q), to_dev(z), to_dev(s)) for q, z, s, _ in parts], to_dev(base.g_idx),
                            [to_dev(b) for _, _, _, b in parts], gs)
    assert mat.info()["N"] == sum(Ns)
    dq = oracle_dq(base)
    w = mat.dequant()
    torch.cuda.synchronize()
    assert np.array_equal(w.cpu().numpy().view(np.uint16), dq.w16)
    for path in ("AUTO", "DECODE", "DECODE_RING", "DECODE_STREAM", "PREFILL"):
        mat.set_path(getattr(q4, "GPTQ_Q4_PATH_" + path))
        for M in (1, 8, 33):
            x = synthetic.activations(M, K, key=(26, K, M))
            y = mat(to_dev(x))
            torch.cuda.synchronize()
            check_y(y, x, dq, base.bias, K, f"fused {path} act={act} M={M}")
            off = 0
            for (q, z, s, b), n in zip(parts, Ns):
                dqi = oracle.dequantize_layer(q, z, s, base.g_idx, K, n, gs)
                check_y(y[:, off:off + n], x, dqi, b, K, f"fused part {off} {path} M={M}")
                off += n
    mat.device_error()
    mat.close()


@pytest.mark.parametrize("K,N,gs,act,fmt,sym", [
    (256, 128, 64, False, 0, False),
    (1024, 448, 32, True, 0, False),
    (1152, 320, 96, True, 1, False),
    (512, 256, -1, False, 0, True),
])
def test_gpu_pack_matches_oracle(q4, K, N, gs, act, fmt, sym):
    """GPU packer against the oracle's packer, bit for bit, on random weights
    plus forced ties (quotients k + 1/2), far out-of-range weights and zero
    points at both ends; then the packed checkpoint through make + matmul."""
    g = np.random.default_rng((27, K, N, act, fmt))
    G = 1 if gs == -1 else K // gs
    geff = K if gs == -1 else gs
    g_idx = (g.permutation(K) // geff).astype(np.int32) if act else None
    scales = g.uniform(0.002, 0.02, (G, N)).astype(np.float16)
    scales[0, :8] = np.float16(0.125)                    # exact quotients for the forced cases
    zeros = None if sym else g.integers(0, 16, (G, N)).astype(np.int32)
    if zeros is not None:
        zeros[0, 0], zeros[0, 1] = 0, 15
    w = g.normal(0, 0.05, (K, N)).astype(np.float16)
    rows0 = np.nonzero((g_idx if act else np.arange(K) // geff) == 0)[0][:8]
    for j, r in enumerate(rows0):
        w[r, :8] = np.float16((j - 3.5) * 0.125)         # quotients -3.5 .. 3.5: ties to even
    w[rows0[0], 8:16] = np.float16(60.0)                  # clamps to 15
    w[rows0[1], 8:16] = np.float16(-60.0)                 # clamps to 0
    qw_ref, qz_ref = oracle.pack(w.view(np.uint16), scales.view(np.uint16), zeros, g_idx, K, N, gs, 1 - fmt)
    qw, qz = q4.pack(to_dev(w), to_dev(scales), None if zeros is None else to_dev(zeros),
                     None if g_idx is None else to_dev(g_idx), gs, fmt)
    torch.cuda.synchronize()
    assert np.array_equal(qw.cpu().numpy(), qw_ref)
    assert np.array_equal(qz.cpu().numpy(), qz_ref)
    mat = q4.Q4Matrix(qw, qz, to_dev(scales), None if g_idx is None else to_dev(g_idx), None, gs)
    mat.set_format(fmt)
    dq = oracle.dequantize_layer(qw_ref, qz_ref, scales, g_idx, K, N, gs, zero_offset=1 - fmt)
    for M in (1, 20):
        x = synthetic.activations(M, K, key=(27, K, N, M))
        y = mat(to_dev(x))
        torch.cuda.synchronize()
        check_y(y, x, dq, None, K, f"packed K={K} N={N} g={gs} act={act} fmt={fmt} M={M}")
    mat.device_error()
