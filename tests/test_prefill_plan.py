"""Host-only checks of the fused prefill's work split (gptq_q4_debug_prefill_plan,
no device call): which tile shape and split each Llama workload gets on a
152-SM GPU, and invariants of the planner over many shapes."""
import os

import pytest

SMS = 152


@pytest.fixture(scope="module")
def q4():
    import __graft_entry__
    b = __graft_entry__._cuda_build_module()
    if not os.path.exists(b.LIB):
        b.build()
    import gptq_bit_weight_gb300
    return gptq_bit_weight_gb300


def plan(q4, M, K, N, sms=SMS):
    return q4.gptq_q4_debug_prefill_plan(M, K, N, sms)


@pytest.mark.parametrize("M,K,N,want", [
    # whole 256 x 256 tiles round robin: the rounds are at least three quarters full
    (2048, 4096, 4096, dict(bm=256, stream_k=0, grid=0)),          # 128 tiles, one round
    (2048, 4096, 11008, dict(bm=256, stream_k=0, grid=0)),         # 344 tiles, rounds 3/4 full
    (2048, 8192, 28672, dict(bm=256, stream_k=0, grid=0)),
    (1024, 28672, 8192, dict(bm=256, stream_k=0, grid=0)),         # 128 tiles
    # even K split: at least two SMs per tile, every piece's CTA sums a share of rows
    (512, 4096, 4096, dict(bm=256, stream_k=1, grid=128, max_pieces=4, piece0_finishes=0)),
    (1024, 4096, 4096, dict(bm=256, stream_k=1, grid=128, max_pieces=2, piece0_finishes=0)),
    (512, 11008, 4096, dict(bm=256, stream_k=1, grid=128, max_pieces=4, piece0_finishes=0)),
    (64, 28672, 8192, dict(bm=128, stream_k=1, grid=128, max_pieces=4, piece0_finishes=0, stage_rows=128)),
    # stream-K ranges, one per SM: piece 0's CTA finishes each cut tile
    (512, 4096, 11008, dict(bm=256, stream_k=1, grid=SMS, piece0_finishes=1)),
    (1024, 8192, 10240, dict(bm=256, stream_k=1, grid=SMS, piece0_finishes=1)),
    (2048, 8192, 10240, dict(bm=256, stream_k=1, grid=SMS, piece0_finishes=1)),   # 320 tiles, rounds 70 % full
    (64, 8192, 28672, dict(bm=128, stream_k=1, grid=SMS, piece0_finishes=1, stage_rows=128)),
    (100, 8192, 28672, dict(bm=128, stream_k=1, grid=SMS, piece0_finishes=1, stage_rows=64)),
    (256, 8192, 28672, dict(bm=256, stream_k=1, grid=SMS, piece0_finishes=1, stage_rows=64)),
])
def test_llama_workloads(q4, M, K, N, want):
    p = plan(q4, M, K, N)
    assert p["bn"] == 256
    for k, v in want.items():
        assert p[k] == v, (M, K, N, k, p)


def tiles_of(p, M, N):
    return ((M + p["bm"] - 1) // p["bm"]) * ((N + 255) // 256)


@pytest.mark.parametrize("sms", [132, 148, 152])
def test_planner_invariants(q4, sms):
    for K in (64, 512, 1024, 4096, 11008 // 64 * 64, 28672):
        for N in (64, 1024, 4096, 10240, 11008, 20416, 28672):
            for M in (1, 17, 100, 128, 129, 256, 300, 512, 1000, 2048, 4096):
                p = plan(q4, M, K, N, sms)
                t = tiles_of(p, M, N)
                KB = K // 64
                assert p["bm"] == (128 if M <= 128 and p["stream_k"] else 256), (M, K, N, p)
                # 128-row stages (x tiles of 64 rows) exactly for M <= 64 off round robin
                assert p["stage_rows"] == (128 if p["stream_k"] and M <= 64 and K % 128 == 0 else 64), (M, K, N, p)
                if not p["stream_k"]:
                    # round robin over 256 x 256 tiles: the rounds at least three quarters full
                    rounds = -(-t // sms)
                    assert p["bm"] == 256 and p["grid"] == 0 and p["max_pieces"] == 1
                    assert 4 * t >= 3 * rounds * sms, (M, K, N, p)
                    continue
                assert 1 <= p["grid"] <= sms, (M, K, N, p)
                if p["piece0_finishes"]:
                    # one range per CTA, fewer than two SMs per tile: a tile spans at
                    # most three CTAs, so its piece 0's CTA adds at most two others
                    assert sms < 2 * t or KB < 16, (M, K, N, p)
                    assert p["max_pieces"] <= 3, (M, K, N, p)
                else:
                    # even split: every tile cut into the same number of equal k ranges
                    assert p["grid"] % t == 0 and p["grid"] // t == p["max_pieces"], (M, K, N, p)
                    assert 2 <= p["max_pieces"] <= 8 and KB // p["max_pieces"] >= 8, (M, K, N, p)


def test_argument_errors(q4):
    for args in ((0, 4096, 4096, SMS), (512, 4000, 4096, SMS), (512, 4096, 4000, SMS), (512, 4096, 4096, 0)):
        with pytest.raises(q4.GPTQ4Error) as e:
            plan(q4, *args)
        assert e.value.status == q4.GPTQ_Q4_INVALID_ARGUMENT
