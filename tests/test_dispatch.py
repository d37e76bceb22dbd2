"""Host-only checks of which kernel a call runs (gptq_q4_debug_dispatch, no
device call): the measured choice of decode kernel for every Llama-70B
projection layer, group size and M up to 16 on a 152-SM GPU, the decode /
prefill threshold, and what each explicit path setting runs."""
import os

import pytest

SMS = 152
R, S, T, P = "decode_reg", "decode_stream", "decode_ring", "prefill"


@pytest.fixture(scope="module")
def q4():
    import __graft_entry__
    b = __graft_entry__._cuda_build_module()
    if not os.path.exists(b.LIB):
        b.build()
    import gptq_bit_weight_gb300
    return gptq_bit_weight_gb300


# AUTO at M = 1, 2, 4, 8, 9, 16, 17: the choices of the measured dispatch
# table (register-streaming / stream-K / TMA-ring per call, CUDA-graph replays
# over more weights than L2) and of the prefill threshold (9 for 32-row
# groups and for 64-row groups on layers of 100 Mi weights or more, else 17).
AUTO_TABLE = {
    (8192, 28672, 32): [R, R, R, R, P, P, P],
    (8192, 28672, 64): [R, R, R, R, P, P, P],
    (8192, 28672, 128): [R, R, R, T, T, T, P],
    (8192, 28672, -1): [R, R, R, T, T, T, P],
    (28672, 8192, 32): [S, S, R, R, P, P, P],
    (28672, 8192, 64): [S, R, R, R, P, P, P],
    (28672, 8192, 128): [S, R, S, S, T, T, P],
    (28672, 8192, -1): [R, R, S, S, T, T, P],
    (8192, 10240, 32): [R, R, R, R, P, P, P],
    (8192, 10240, 64): [R, R, R, R, T, T, P],
    (8192, 10240, 128): [R, R, R, T, T, T, P],
    (8192, 10240, -1): [R, R, R, T, T, T, P],
}


@pytest.mark.parametrize("K,N,g", sorted(AUTO_TABLE))
def test_auto_matches_the_measured_table(q4, K, N, g):
    got = [q4.gptq_q4_debug_dispatch(M, K, N, g, q4.GPTQ_Q4_PATH_AUTO, SMS) for M in (1, 2, 4, 8, 9, 16, 17)]
    assert got == AUTO_TABLE[(K, N, g)]


@pytest.mark.parametrize("K,N", [(4096, 4096), (4096, 11008), (11008, 4096), (4096, 12288)])
def test_llama7b_decode(q4, K, N):
    """Layers below 64 Mi weights: the register-streaming kernel up to eight
    rows (on 11008 x 4096 too: tall, but under 100 Mi weights, so no stream-K);
    at 9-16 rows the TMA ring, except below 24 Mi weights (4096 x 4096)."""
    for M in (1, 2, 4, 8):
        assert q4.gptq_q4_debug_dispatch(M, K, N, 128, q4.GPTQ_Q4_PATH_AUTO, SMS) == R
    assert q4.gptq_q4_debug_dispatch(16, K, N, 128, q4.GPTQ_Q4_PATH_AUTO, SMS) == (R if K * N < 24 << 20 else T)


def test_explicit_paths(q4):
    K, N, g = 4096, 11008, 128
    for M in (1, 8, 16, 17, 300):
        assert q4.gptq_q4_debug_dispatch(M, K, N, g, q4.GPTQ_Q4_PATH_PREFILL, SMS) == P
        assert q4.gptq_q4_debug_dispatch(M, K, N, g, q4.GPTQ_Q4_PATH_DECODE_MMA, SMS) == R
        # the stream-K decode takes at most eight rows, the TMA ring at most 16
        assert q4.gptq_q4_debug_dispatch(M, K, N, g, q4.GPTQ_Q4_PATH_DECODE_STREAM, SMS) == (S if M <= 8 else R)
        assert q4.gptq_q4_debug_dispatch(M, K, N, g, q4.GPTQ_Q4_PATH_DECODE_RING, SMS) == (T if M <= 16 else R)
    # the tcgen05 decode where its planner accepts the shape, else the default decode kernel
    assert q4.gptq_q4_debug_dispatch(1, K, N, g, q4.GPTQ_Q4_PATH_DECODE_TC, SMS) in ("decode_tc", R)
    assert q4.gptq_q4_debug_dispatch(300, K, N, g, q4.GPTQ_Q4_PATH_DECODE_TC, SMS) == R


def test_threshold_invariants(q4):
    """AUTO never runs the fused prefill below 9 rows and always from 17."""
    for K in (1024, 4096, 8192, 28672):
        for N in (1024, 4096, 10240, 28672):
            for g in (32, 64, 128, -1):
                for M in range(1, 9):
                    assert q4.gptq_q4_debug_dispatch(M, K, N, g, q4.GPTQ_Q4_PATH_AUTO, SMS) != P
                for M in (17, 64, 512):
                    assert q4.gptq_q4_debug_dispatch(M, K, N, g, q4.GPTQ_Q4_PATH_AUTO, SMS) == P


def test_argument_errors(q4):
    bad = [(0, 4096, 4096, 128, 0), (1, 4000, 4096, 128, 0), (1, 4096, 4000, 128, 0), (1, 4096, 4096, 48, 0),
           (1, 4096, 4096, 100, 0), (1, 4096, 4096, 128, 9), (1, 4096, 4096, 128, -1)]
    for M, K, N, g, path in bad:
        with pytest.raises(q4.GPTQ4Error) as e:
            q4.gptq_q4_debug_dispatch(M, K, N, g, path, SMS)
        assert e.value.status == q4.GPTQ_Q4_INVALID_ARGUMENT
    with pytest.raises(q4.GPTQ4Error):
        q4.gptq_q4_debug_dispatch(1, 4096, 4096, 128, 0, 0)
