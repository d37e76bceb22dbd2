"""Full-size parity on the Llama-70B-shaped sweep (sweep_70b): every (K, N),
groupsize and act-order combination at full size on the GPU, with the oracle
evaluated on a seeded sample of 8-column blocks (a block is one qzeros word,
so the oracle runs on exactly those columns of the real tensors) and, for
the largest M, a seeded row sample.  Every M of the workload runs on every
layer configuration through the default path; M = 16 and 64 also run the
decode and prefill paths forced."""
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


def column_sample(layer, nblocks, seed):
    g = np.random.default_rng(seed)
    blocks = np.sort(g.choice(layer.N // 8, size=nblocks, replace=False))
    blocks[0] = 0
    blocks[-1] = layer.N // 8 - 1
    blocks = np.unique(blocks)
    cols = (blocks[:, None] * 8 + np.arange(8)[None, :]).reshape(-1)
    dq = oracle.dequantize_layer(layer.qweight[:, cols], layer.qzeros[:, blocks], layer.scales[:, cols],
                                 layer.g_idx, layer.K, cols.size, layer.groupsize)
    return cols, dq


CASES = [(K, N, g, a) for (K, N) in synthetic.SWEEP_70B_SHAPES for g in synthetic.SWEEP_70B_G for a in (False, True)]


@pytest.mark.parametrize("K,N,gs,act", CASES)
def test_sweep_70b_sampled(q4, K, N, gs, act):
    layer = synthetic.workload_layer("sweep_70b", K, N, gs, act)
    mat = q4.Q4Matrix(to_dev(layer.qweight), to_dev(layer.qzeros), to_dev(layer.scales), to_dev(layer.g_idx),
                      None, gs)
    cols, dq = column_sample(layer, 12, seed=K + N + (gs & 0xFFFF) + act)
    tcols = torch.from_numpy(cols).to(DEV)
    # unpacked codes and dequantized weights: bit-exact on the sampled columns
    q_gpu, _ = mat.debug_unpack()
    w_gpu = mat.dequant()
    torch.cuda.synchronize()
    assert np.array_equal(q_gpu[:, tcols].cpu().numpy(), dq.q)
    assert np.array_equal(w_gpu[:, tcols].cpu().numpy().view(np.uint16), dq.w16)
    del q_gpu, w_gpu
    for M in synthetic.SWEEP_70B_M:
        x = synthetic.workload_x("sweep_70b", K, N, gs, act, M)
        xd = to_dev(x)
        rows = np.arange(M) if M <= 256 else np.unique(np.concatenate(
            [[0, M - 1], np.random.default_rng(M).choice(M, 14, replace=False)]))
        y_ref = oracle.reference_output(x[rows], dq)
        tol = oracle.tolerance(x, dq.w16, y_ref, K)
        paths = [q4.GPTQ_Q4_PATH_AUTO]
        if M in (16, 64):
            paths += [q4.GPTQ_Q4_PATH_DECODE, q4.GPTQ_Q4_PATH_PREFILL]
        for path in paths:
            mat.set_path(path)
            y = mat(xd)
            torch.cuda.synchronize()
            got = y[torch.from_numpy(rows).to(DEV)][:, tcols].float().cpu().numpy().astype(np.float64)
            err = np.abs(got - y_ref)
            assert np.all(err <= tol), (f"{K}x{N} g={gs} act={act} M={M} path={path}: worst err/tol "
                                        f"{float(np.max(err / tol)):.3f}")
    mat.set_path(q4.GPTQ_Q4_PATH_AUTO)
    mat.device_error()
    mat.close()
