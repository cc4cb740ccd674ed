"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Buffers, plans and control-plane state must match bit for bit; GEMM outputs
within |gpu - oracle| <= 2e-2 + 1e-2 |oracle| elementwise.  Inputs change
every round (seed*1000 + round) so a stale read of an earlier round fails.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from consumer_movement_gemm_gb300 import tovl
from tests.gpu_util import assert_close, bits

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _build():
    from consumer_movement_gemm_gb300 import build
    build.build()
    oracle.build()


def _handle(**kw):
    kw.setdefault("max_rows", 1 << 14)
    kw.setdefault("max_pairs", 1 << 14)
    kw.setdefault("max_experts", 64)
    kw.setdefault("wait_timeout_ns", 2_000_000_000)
    return tovl.Handle(0, **kw)


def _check_ctrl(h, R):
    slots, cnts, rb, seq = h.read_ctrl()
    o_slots, o_cnts, o_rb = oracle.ctrl_state(R, slots.size, rb.size)
    assert seq == R
    assert np.array_equal(slots, o_slots), "slots"
    assert np.array_equal(cnts, o_cnts), "chunk counters"
    assert np.array_equal(rb, o_rb), "row-block counters"


# ------------------------------------------------------------------ GEMM alone
@pytest.mark.parametrize("M,K,N", [(256, 256, 256), (128, 512, 512)])
@pytest.mark.parametrize("pairs", [1, 0])
def test_gemm_only_identity_is_exact(M, K, N, pairs):
    with _handle() as h:
        h.set_option(tovl.OPT_PAIRS, pairs)
        A = workloads.bf16_normal((M, K), 1.0, 11, DEV)
        W = torch.zeros(K, N, dtype=torch.bfloat16, device=DEV)
        idx = torch.arange(min(K, N), device=DEV)
        W[idx, idx] = 1.0
        out = torch.full((M, N), 7.0, dtype=torch.bfloat16, device=DEV)
        h.gemm_only(A, W, out)
        assert h.sync_status() == 0
        want = torch.zeros(M, N, dtype=torch.bfloat16, device=DEV)
        want[:, :min(K, N)] = A[:, :min(K, N)]
        assert torch.equal(out, want)


@pytest.mark.parametrize("M,K,N", [(384, 320, 512), (300, 192, 256), (1, 64, 256), (640, 1024, 768)])
@pytest.mark.parametrize("pairs", [1, 0])
def test_gemm_only_matches_oracle(M, K, N, pairs):
    with _handle() as h:
        h.set_option(tovl.OPT_PAIRS, pairs)
        A = workloads.bf16_normal((M, K), 1 / math.sqrt(K), 12, DEV)
        W = workloads.bf16_normal((K, N), 1 / math.sqrt(K), 13, DEV)
        out = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
        h.gemm_only(A, W, out)
        assert h.sync_status() == 0
        assert_close(out, oracle.matmul_f32(bits(A), bits(W)), "gemm_only")


# ------------------------------------------------------------------ gather + GEMM
def _gather_round(h, cfg, seed):
    X, W = workloads.gather_inputs(cfg, seed, DEV)
    gathered = torch.empty(cfg.M, cfg.K, dtype=torch.bfloat16, device=DEV)
    out = torch.empty(cfg.M, cfg.N, dtype=torch.bfloat16, device=DEV)
    h.gather_gemm(X, W, gathered, out)
    return X, W, gathered, out


@pytest.mark.parametrize("k_slices", [1, 2, 4, 8])
@pytest.mark.parametrize("pairs", [1, 0])
@pytest.mark.parametrize("mode", [0, 1])
def test_tiny_gather_gemm_three_rounds(k_slices, pairs, mode):
    cfg = workloads.TINY
    with _handle(k_slices=k_slices) as h:
        h.set_option(tovl.OPT_PAIRS, pairs)
        h.set_option(tovl.OPT_PRODUCER_MODE, mode)
        if pairs:
            assert h.get_option(tovl.OPT_PAIRS) == 1, "CTA pairs unavailable on this device"
        for r in range(1, cfg.rounds + 1):
            X, W, gathered, out = _gather_round(h, cfg, workloads.round_seed(cfg.seed, r))
            assert h.sync_status() == 0
            shards = [bits(X[s]) for s in range(cfg.shards)]
            G = oracle.gather(shards)
            assert np.array_equal(bits(gathered), G), f"gathered buffer, round {r}"
            assert_close(out, oracle.matmul_f32(G, bits(W)), f"round {r}")
            _check_ctrl(h, r)


# item shapes: (3,100,192) 32-row items; (1,64,64) 64-row items; (2,70,8192,KS=1)
# single-row items wider than one 8 KB pass; (3,150,1024) and (2,300,2048,KS=2)
# 4-row items with 8 lanes per row
@pytest.mark.parametrize("S,R,K,N,P,KS", [(3, 100, 192, 256, 4, 2), (1, 64, 64, 512, 1, 4), (5, 77, 128, 256, 32, 1),
                                          (2, 200, 320, 256, 8, 4), (7, 33, 448, 512, 3, 8),
                                          (2, 70, 8192, 256, 4, 1), (3, 150, 1024, 256, 4, 1),
                                          (2, 300, 2048, 512, 6, 2)])
@pytest.mark.parametrize("pairs", [1, 0])
@pytest.mark.parametrize("mode", [0, 1])
def test_gather_gemm_ragged(S, R, K, N, P, KS, pairs, mode):
    cfg = workloads.GatherCfg("ragged", S, R, K, N, rounds=2)
    with _handle(producer_ctas=P, k_slices=KS) as h:
        h.set_option(tovl.OPT_PAIRS, pairs)
        h.set_option(tovl.OPT_PRODUCER_MODE, mode)
        for r in range(1, 3):
            X, W, gathered, out = _gather_round(h, cfg, 100 + r)
            assert h.sync_status() == 0
            G = oracle.gather([bits(X[s]) for s in range(S)])
            assert np.array_equal(bits(gathered), G)
            assert_close(out, oracle.matmul_f32(G, bits(W)), "ragged")
            _check_ctrl(h, r)


@pytest.mark.parametrize("S,R,K,N,KS", [(4, 96, 256, 512, 4), (3, 100, 192, 256, 2)])
@pytest.mark.parametrize("pairs", [1, 0])
def test_gather_gemm_embedded_copy_warps(S, R, K, N, KS, pairs):
    # option 18 = 2: the gather too runs without producer CTAs, its rows copied
    # by the consumer CTAs' spare warps (the kernels with embedded producers,
    # pair and single-CTA, in gather mode)
    cfg = workloads.GatherCfg("embedded", S, R, K, N, rounds=3)
    with _handle(k_slices=KS) as h:
        h.set_option(tovl.OPT_PAIRS, pairs)
        h.set_option(tovl.OPT_EMBEDDED, 2)
        for r in range(1, 4):
            X, W, gathered, out = _gather_round(h, cfg, 200 + r)
            assert h.sync_status() == 0
            assert h.get_option(tovl.OPT_PRODUCERS) == 0
            G = oracle.gather([bits(X[s]) for s in range(S)])
            assert np.array_equal(bits(gathered), G)
            assert_close(out, oracle.matmul_f32(G, bits(W)), "embedded gather")
            _check_ctrl(h, r)


@pytest.mark.parametrize("k_slices", [1, 4])
def test_copy_only_control(k_slices):
    cfg = workloads.GatherCfg("copy", 4, 96, 256, 256, rounds=2)
    with _handle(k_slices=k_slices) as h:
        for r in range(1, 3):
            X, _ = workloads.gather_inputs(cfg, r, DEV)
            gathered = torch.empty(cfg.M, cfg.K, dtype=torch.bfloat16, device=DEV)
            h.copy_only(X, gathered)
            assert h.sync_status() == 0
            assert np.array_equal(bits(gathered), oracle.gather([bits(X[s]) for s in range(4)]))
            _check_ctrl(h, r)


@pytest.mark.parametrize("pairs", [1, 0])
def test_timeout_is_reported_and_handle_recovers(pairs):
    cfg = workloads.TINY
    with _handle(wait_timeout_ns=5_000_000, k_slices=2) as h:
        h.set_option(tovl.OPT_PAIRS, pairs)
        h.set_option(tovl.OPT_FAULT_GATE_OFFSET, 1)      # gates wait for a sequence nobody publishes
        _gather_round(h, cfg, 1)
        assert h.sync_status() == tovl.TOVL_ERR_TIMEOUT
        assert h.sync_status() == 0                        # the status word was cleared
        h.set_option(tovl.OPT_FAULT_GATE_OFFSET, 0)
        X, W, gathered, out = _gather_round(h, cfg, 2)
        assert h.sync_status() == 0
        G = oracle.gather([bits(X[s]) for s in range(cfg.shards)])
        assert np.array_equal(bits(gathered), G)
        assert_close(out, oracle.matmul_f32(G, bits(W)), "after timeout")
        _check_ctrl(h, 2)


# ------------------------------------------------------------------ dispatch + grouped GEMM
def _dispatch_round(h, x, topk_np, W):
    T, H = x.shape
    k = topk_np.shape[1]
    E, _, N = W.shape
    rows = tovl.dispatch_rows(T, k, E)
    topk = torch.from_numpy(topk_np).to(DEV)
    dispatched = torch.full((rows, H), 3.0, dtype=torch.bfloat16, device=DEV)   # non-zero garbage
    offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    out = torch.empty(rows, N, dtype=torch.bfloat16, device=DEV)
    h.dispatch_grouped_gemm(x, topk, W, dispatched, offs, out)
    return dispatched, offs, out


def _check_dispatch(h, x, topk_np, W, dispatched, offs, out, R):
    T, H = x.shape
    k = topk_np.shape[1]
    E = W.shape[0]
    p = oracle.dispatch_plan(topk_np, E)
    counts, dst, src, pad, blk, m_pad = h.read_plan(T, k, E)
    assert m_pad == p.m_pad
    assert np.array_equal(counts, p.counts)
    assert np.array_equal(offs.cpu().numpy(), p.off)
    assert np.array_equal(dst, p.dst)
    assert np.array_equal(src, p.src)
    assert np.array_equal(pad, p.pad)
    assert np.array_equal(blk, p.blk_e)
    D = oracle.dispatch(bits(x), p.dst, k, p.m_pad)
    assert np.array_equal(bits(dispatched[:p.m_pad]), D), "dispatched buffer"
    O = oracle.grouped_matmul_f32(D, bits(W), p.off)
    assert_close(out[:p.m_pad], O, "grouped GEMM")
    assert torch.count_nonzero(out[:p.m_pad][torch.from_numpy(p.src < 0).to(DEV)]) == 0
    _check_ctrl(h, R)


ROUTINGS = {
    "uniform": lambda s: (workloads.uniform_topk(300, 2, 5, s), 5),
    "zipf": lambda s: (workloads.zipf_topk(700, 4, 12, 1.2, s), 12),
    "all_to_one": lambda s: (workloads.all_to_one_topk(260, 3, 1), 3),
    "empty_expert": lambda s: (workloads.uniform_topk(200, 2, 4, s), 7),
}


@pytest.mark.parametrize("routing", list(ROUTINGS))
@pytest.mark.parametrize("k_slices", [1, 2])
@pytest.mark.parametrize("mode,switch", [(0, 1), (1, 1), (0, 0)])
def test_dispatch_grouped_gemm_small(routing, k_slices, mode, switch):
    # switch: tiles from the ticket counter and producer CTAs that turn
    # consumer (1), or the static schedule (0)
    H, N = 192, 256
    with _handle(k_slices=k_slices) as h:
        h.set_option(tovl.OPT_EMBEDDED, 0)      # producer CTAs (the embedded copy has its own test)
        h.set_option(tovl.OPT_PRODUCER_MODE, mode)
        h.set_option(tovl.OPT_ROLE_SWITCH, switch)
        for r in range(1, 4):
            topk_np, E = ROUTINGS[routing](workloads.round_seed(1, r))
            T = topk_np.shape[0]
            x = workloads.bf16_normal((T, H), 1 / math.sqrt(H), 200 + r, DEV)
            W = workloads.bf16_normal((E, H, N), 1 / math.sqrt(H), 300 + r, DEV)
            dispatched, offs, out = _dispatch_round(h, x, topk_np, W)
            assert h.sync_status() == 0
            _check_dispatch(h, x, topk_np, W, dispatched, offs, out, r)


@pytest.mark.parametrize("routing", list(ROUTINGS))
@pytest.mark.parametrize("switch", [1, 2])
def test_dispatch_pair_tiles_on_256_row_segments(routing, switch):
    # option 17: segments aligned to 256 rows, CTA-pair tiles; the layout is
    # the oracle's plan with 256-row blocks, the counters stay per 128 rows.
    # switch 1: fixed pair roles; 2: one ticket per pair, producer pairs join
    H, N = 192, 512
    with _handle(k_slices=2) as h:
        h.set_option(tovl.OPT_EMBEDDED, 0)      # producer CTAs (the embedded copy has its own test)
        h.set_option(tovl.OPT_DISPATCH_ALIGN, 256)
        h.set_option(tovl.OPT_ROLE_SWITCH, switch)
        for r in range(1, 4):
            topk_np, E = ROUTINGS[routing](workloads.round_seed(3, r))
            T, k = topk_np.shape
            x = workloads.bf16_normal((T, H), 1 / math.sqrt(H), 900 + r, DEV)
            W = workloads.bf16_normal((E, H, N), 1 / math.sqrt(H), 950 + r, DEV)
            rows = tovl.dispatch_rows_aligned(T, k, E, 256)
            dispatched = torch.full((rows, H), 3.0, dtype=torch.bfloat16, device=DEV)
            offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
            out = torch.empty(rows, N, dtype=torch.bfloat16, device=DEV)
            h.dispatch_grouped_gemm(x, torch.from_numpy(topk_np).to(DEV), W, dispatched, offs, out)
            assert h.sync_status() == 0
            p = oracle.dispatch_plan(topk_np, E, block_rows=256)
            counts, dst, src, pad, blk, m_pad = h.read_plan(T, k, E)
            assert m_pad == p.m_pad and m_pad % 256 == 0
            assert np.array_equal(offs.cpu().numpy(), p.off)
            assert np.array_equal(dst, p.dst)
            assert np.array_equal(src, p.src)
            # per 128-row block: padding = rows without a source, expert = segment
            real = (p.src >= 0).reshape(-1, 128).sum(axis=1)
            assert np.array_equal(pad, 128 - real)
            assert np.array_equal(blk, np.searchsorted(p.off, np.arange(0, m_pad, 128), side="right") - 1)
            D = oracle.dispatch(bits(x), p.dst, k, p.m_pad)
            assert np.array_equal(bits(dispatched[:m_pad]), D), "dispatched buffer"
            assert_close(out[:m_pad], oracle.grouped_matmul_f32(D, bits(W), p.off), "grouped GEMM, pair tiles")
            _check_ctrl(h, r)


def test_dispatch_bad_expert_id_is_a_noop_round():
    H, N, E = 64, 256, 3
    with _handle() as h:
        topk_np = np.array([[0, 1], [2, 5]], np.int32)
        x = workloads.bf16_normal((2, H), 1.0, 1, DEV)
        W = workloads.bf16_normal((E, H, N), 1.0, 2, DEV)
        _, offs, _ = _dispatch_round(h, x, topk_np, W)
        assert h.sync_status() == tovl.TOVL_ERR_INVALID
        assert torch.count_nonzero(offs) == 0
        _check_ctrl(h, 1)
        # the next round is normal
        topk_np = np.array([[0, 1], [2, 1]], np.int32)
        dispatched, offs, out = _dispatch_round(h, x, topk_np, W)
        assert h.sync_status() == 0
        _check_dispatch(h, x, topk_np, W, dispatched, offs, out, 2)


# ------------------------------------------------------------------ combine
def _combine_round(h, rows, N, T, k, seed):
    y = workloads.bf16_normal((rows, N), 1.0, seed, DEV)
    w_np = workloads.gate_weights(T, k, seed + 1)
    w = torch.from_numpy(w_np).to(DEV)
    staging = torch.full((max(T * k, 1), N), 5.0, dtype=torch.bfloat16, device=DEV)
    combined = torch.full((max(T, 1), N), 5.0, dtype=torch.bfloat16, device=DEV)
    h.combine(y, w, staging, combined)
    return y, w_np, staging, combined


@pytest.mark.parametrize("routing", list(ROUTINGS))
@pytest.mark.parametrize("mode,pdl,emb", [(0, 1, 1), (0, 0, 1), (0, 1, 0), (1, 1, 0)])
def test_combine_after_dispatch(routing, mode, pdl, emb):
    # combine runs on a seeded expert-output tensor, so staging and combined
    # rows are compared bit for bit with the oracle's; plan -> fused kernel ->
    # combine run with and without programmatic dependent launches; emb 1 (the
    # default): every CTA copies and reduces, 0: producer and reducer CTAs
    # (vector or staged copies)
    H, N = 128, 320
    with _handle(k_slices=2) as h:
        h.set_option(tovl.OPT_EMBEDDED, emb)
        h.set_option(tovl.OPT_PRODUCER_MODE, mode)
        h.set_option(tovl.OPT_PDL, pdl)
        assert h.get_option(tovl.OPT_PDL) == pdl
        R = 0
        for r in range(1, 4):
            topk_np, E = ROUTINGS[routing](workloads.round_seed(2, r))
            T, k = topk_np.shape
            x = workloads.bf16_normal((T, H), 1 / math.sqrt(H), 400 + r, DEV)
            W = workloads.bf16_normal((E, H, 256), 1 / math.sqrt(H), 500 + r, DEV)
            _dispatch_round(h, x, topk_np, W)
            R += 1
            rows = tovl.dispatch_rows(T, k, E)
            y, w_np, staging, combined = _combine_round(h, rows, N, T, k, 600 + r)
            R += 1
            assert h.sync_status() == 0
            p = oracle.dispatch_plan(topk_np, E)
            S, C = oracle.combine(bits(y), p.dst, w_np)
            assert np.array_equal(bits(staging[:T * k]), S), "staging"
            assert np.array_equal(bits(combined[:T]), C), "combined"
            _check_ctrl(h, R)


def test_combine_after_pair_tile_dispatch():
    # the 256-row segment layout changes where expert rows live, not combine
    H, N, T, k, E = 128, 256, 300, 2, 5
    with _handle() as h:
        h.set_option(tovl.OPT_DISPATCH_ALIGN, 256)
        topk_np = workloads.uniform_topk(T, k, E, 31)
        x = workloads.bf16_normal((T, H), 1.0, 32, DEV)
        W = workloads.bf16_normal((E, H, 256), 1.0, 33, DEV)
        rows = tovl.dispatch_rows_aligned(T, k, E, 256)
        dispatched = torch.zeros(rows, H, dtype=torch.bfloat16, device=DEV)
        offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
        out = torch.empty(rows, 256, dtype=torch.bfloat16, device=DEV)
        h.dispatch_grouped_gemm(x, torch.from_numpy(topk_np).to(DEV), W, dispatched, offs, out)
        y, w_np, staging, combined = _combine_round(h, rows, N, T, k, 34)
        assert h.sync_status() == 0
        S, C = oracle.combine(bits(y), oracle.dispatch_plan(topk_np, E, block_rows=256).dst, w_np)
        assert np.array_equal(bits(staging[:T * k]), S)
        assert np.array_equal(bits(combined[:T]), C)
        _check_ctrl(h, 2)


@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (21, 3, 5), (64, 1, 2), (100, 8, 16)])
def test_combine_shapes(T, k, E):
    # one token; tokens straddling 64-row chunks (k=3); exactly one chunk;
    # k=8 with a ragged last chunk
    H, N = 64, 64
    with _handle() as h:
        topk_np = workloads.uniform_topk(T, k, E, 9)
        x = workloads.bf16_normal((T, H), 1.0, 1, DEV)
        W = workloads.bf16_normal((E, H, 256), 1.0, 2, DEV)
        _dispatch_round(h, x, topk_np, W)
        y, w_np, staging, combined = _combine_round(h, tovl.dispatch_rows(T, k, E), N, T, k, 3)
        assert h.sync_status() == 0
        S, C = oracle.combine(bits(y), oracle.dispatch_plan(topk_np, E).dst, w_np)
        assert np.array_equal(bits(staging[:T * k]), S)
        assert np.array_equal(bits(combined[:T]), C)
        _check_ctrl(h, 2)


@pytest.mark.parametrize("T,k,E", [(40, 67, 8), (9, 130, 5), (3, 2100, 4)])
def test_combine_tokens_spanning_many_chunks(T, k, E):
    # a token's k staged rows span three or more 64-row chunks (k = 67, 130),
    # and more than 32 of them (k = 2100): the reducer must wait on every one
    # of those chunk slots, not only the first and the last.  Experts are
    # drawn with replacement, so a token may name one expert many times.
    H, N = 64, 128
    with _handle(max_rows=1 << 14, max_pairs=1 << 14) as h:
        for r in (1, 2):
            topk_np = workloads.repeated_topk(T, k, E, workloads.round_seed(7, r))
            x = workloads.bf16_normal((T, H), 1.0, 70 + r, DEV)
            W = workloads.bf16_normal((E, H, 256), 1.0, 80 + r, DEV)
            _dispatch_round(h, x, topk_np, W)
            y, w_np, staging, combined = _combine_round(h, tovl.dispatch_rows(T, k, E), N, T, k, 90 + r)
            assert h.sync_status() == 0
            S, C = oracle.combine(bits(y), oracle.dispatch_plan(topk_np, E).dst, w_np)
            assert np.array_equal(bits(staging[:T * k]), S), f"staging, round {r}"
            assert np.array_equal(bits(combined[:T]), C), f"combined, round {r}"
            _check_ctrl(h, 2 * r)


def test_moe_layer_dispatch_gemm_combine():
    # the whole layer against the oracle's: dispatch, grouped GEMM, combine
    T, H, k, E, N = 300, 256, 2, 6, 512
    with _handle() as h:
        topk_np = workloads.uniform_topk(T, k, E, 21)
        x = workloads.bf16_normal((T, H), 1 / math.sqrt(H), 22, DEV)
        W = workloads.bf16_normal((E, H, N), 1 / math.sqrt(H), 23, DEV)
        dispatched, offs, out = _dispatch_round(h, x, topk_np, W)
        w_np = workloads.gate_weights(T, k, 24)
        staging = torch.empty(T * k, N, dtype=torch.bfloat16, device=DEV)
        combined = torch.empty(T, N, dtype=torch.bfloat16, device=DEV)
        h.combine(out, torch.from_numpy(w_np).to(DEV), staging, combined)
        assert h.sync_status() == 0
        p = oracle.dispatch_plan(topk_np, E)
        D = oracle.dispatch(bits(x), p.dst, k, p.m_pad)
        Y = oracle.f32_to_bf16(oracle.grouped_matmul_f32(D, bits(W), p.off))
        _, C = oracle.combine(Y, p.dst, w_np)
        assert_close(combined, oracle.bf16_to_f32(C), "combined layer")
        _check_ctrl(h, 2)


def test_combine_timeout_and_rejected_plan():
    H, N = 64, 64
    with _handle(wait_timeout_ns=5_000_000) as h:
        topk_np = workloads.uniform_topk(50, 2, 4, 5)
        x = workloads.bf16_normal((50, H), 1.0, 1, DEV)
        W = workloads.bf16_normal((4, H, 256), 1.0, 2, DEV)
        _dispatch_round(h, x, topk_np, W)
        h.set_option(tovl.OPT_FAULT_GATE_OFFSET, 1)      # reducers wait for a sequence nobody publishes
        _combine_round(h, tovl.dispatch_rows(50, 2, 4), N, 50, 2, 3)
        assert h.sync_status() == tovl.TOVL_ERR_TIMEOUT
        h.set_option(tovl.OPT_FAULT_GATE_OFFSET, 0)
        y, w_np, staging, combined = _combine_round(h, tovl.dispatch_rows(50, 2, 4), N, 50, 2, 4)
        assert h.sync_status() == 0
        S, C = oracle.combine(bits(y), oracle.dispatch_plan(topk_np, 4).dst, w_np)
        assert np.array_equal(bits(combined[:50]), C)
        _check_ctrl(h, 3)
        # a rejected plan makes the next combine a no-op round that reports it
        bad = np.array([[0, 1], [2, 9]], np.int32)
        _dispatch_round(h, x[:2], bad, W)
        assert h.sync_status() == tovl.TOVL_ERR_INVALID
        _combine_round(h, 256, N, 2, 2, 5)
        assert h.sync_status() == tovl.TOVL_ERR_INVALID
        _check_ctrl(h, 5)


# ------------------------------------------------------------------ GEMM + reduce-scatter
def _rs_round(h, S, M, Ks, N, seed):
    X = workloads.bf16_normal((S, M, Ks), 1 / math.sqrt(S * Ks), seed, DEV)
    W = workloads.bf16_normal((S, Ks, N), 1.0, seed + 1, DEV)
    partials = torch.full((S, M, N), 3.0, dtype=torch.bfloat16, device=DEV)
    out = torch.full((M, N), 3.0, dtype=torch.bfloat16, device=DEV)
    h.gemm_reduce_scatter(X, W, partials, out)
    return X, W, partials, out


@pytest.mark.parametrize("S,M,Ks,N,P", [(4, 512, 256, 512, 0), (1, 256, 128, 256, 0), (3, 384, 192, 768, 4),
                                        (5, 128, 64, 256, 8), (2, 1024, 512, 1024, 16)])
@pytest.mark.parametrize("pairs", [1, 0])
def test_gemm_reduce_scatter(S, M, Ks, N, P, pairs):
    # (3, 384): an odd number of row blocks runs single-CTA tiles even with pairs on
    with _handle(producer_ctas=P, k_slices=4) as h:
        h.set_option(tovl.OPT_PAIRS, pairs)
        for r in range(1, 3):
            X, W, partials, out = _rs_round(h, S, M, Ks, N, 700 + r)
            assert h.sync_status() == 0
            Po, Oo = oracle.gemm_reduce_scatter(bits(X), bits(W))
            for s in range(S):
                assert_close(partials[s], oracle.bf16_to_f32(Po[s]), f"partial {s}")
            assert_close(out, oracle.bf16_to_f32(Oo), "reduced")
            _check_ctrl(h, r)


@pytest.mark.parametrize("S,M,Ks,N", [(4, 512, 256, 512), (3, 384, 192, 768), (5, 256, 64, 256),
                                      (40, 256, 64, 256), (2, 1024, 512, 1024)])
@pytest.mark.parametrize("epi", [1, 0])
def test_gemm_reduce_scatter_reducer_placement(S, M, Ks, N, epi):
    # epi 1: the computer of shard (o mod S)'s partial of output tile o sums
    # the tile in its idle warps, no producer CTAs; epi 0 (the default):
    # producer CTAs reduce.  S = 40 makes a reducer poll more than 32 slots.
    with _handle(k_slices=2) as h:
        h.set_option(tovl.OPT_RS_EPILOGUE, epi)
        for r in range(1, 3):
            X, W, partials, out = _rs_round(h, S, M, Ks, N, 900 + r)
            assert h.sync_status() == 0
            if epi:
                assert h.get_option(tovl.OPT_PRODUCERS) == 0, "the epilogue reduction launches no producer CTAs"
            Po, Oo = oracle.gemm_reduce_scatter(bits(X), bits(W))
            for s in range(S):
                assert_close(partials[s], oracle.bf16_to_f32(Po[s]), f"partial {s}")
            assert_close(out, oracle.bf16_to_f32(Oo), "reduced")
            _check_ctrl(h, r)


@pytest.mark.parametrize("S,M,Ks,N,P", [(4, 512, 256, 512, 0), (3, 384, 192, 768, 4)])
def test_gemm_reduce_scatter_without_role_switch(S, M, Ks, N, P):
    with _handle(producer_ctas=P, k_slices=4) as h:
        h.set_option(tovl.OPT_ROLE_SWITCH, 0)
        h.set_option(tovl.OPT_RS_EPILOGUE, 0)
        for r in range(1, 3):
            X, W, partials, out = _rs_round(h, S, M, Ks, N, 800 + r)
            assert h.sync_status() == 0
            _, Oo = oracle.gemm_reduce_scatter(bits(X), bits(W))
            assert_close(out, oracle.bf16_to_f32(Oo), "reduced")
            _check_ctrl(h, r)


def test_gemm_reduce_scatter_timeout_recovers():
    with _handle(wait_timeout_ns=5_000_000, k_slices=2) as h:
        h.set_option(tovl.OPT_FAULT_GATE_OFFSET, 1)      # reducers wait for a sequence nobody publishes
        _rs_round(h, 2, 256, 128, 256, 1)
        assert h.sync_status() == tovl.TOVL_ERR_TIMEOUT
        h.set_option(tovl.OPT_FAULT_GATE_OFFSET, 0)
        X, W, partials, out = _rs_round(h, 2, 256, 128, 256, 2)
        assert h.sync_status() == 0
        _, Oo = oracle.gemm_reduce_scatter(bits(X), bits(W))
        assert_close(out, oracle.bf16_to_f32(Oo), "after timeout")
        _check_ctrl(h, 2)


def test_gemm_reduce_scatter_rejects_shapes():
    with _handle() as h:
        X = torch.zeros(2, 100, 64, dtype=torch.bfloat16, device=DEV)
        W = torch.zeros(2, 64, 256, dtype=torch.bfloat16, device=DEV)
        P = torch.zeros(2, 100, 256, dtype=torch.bfloat16, device=DEV)
        O = torch.zeros(100, 256, dtype=torch.bfloat16, device=DEV)
        with pytest.raises(tovl.TovlError):
            h.gemm_reduce_scatter(X, W, P, O)                # M not a multiple of 128
        assert h.sync_status() == 0
        _check_ctrl(h, 0)


# ------------------------------------------------------------------ gated copy
@pytest.mark.parametrize("row_bytes", [256, 1024, 8192])
@pytest.mark.parametrize("copy_mode", [tovl.TOVL_COPY_VECTOR, tovl.TOVL_COPY_BULK])
@pytest.mark.parametrize("n", [5000, 100, 20000])
def test_gated_copy_small(row_bytes, copy_mode, n):
    # 100 rows: most bulk issuer warps get no row; 20000 rows: about 33 rows per
    # issuer, so every issuer counts one full batch of 32 retired rows and a
    # partial one
    with _handle(copy_mode=copy_mode, max_rows=n, k_slices=2) as h:
        for r in range(1, 3):
            perm_np = workloads.permutation(n, r)
            src = workloads.random_bytes(n, row_bytes, r, DEV)
            dst = torch.zeros_like(src)
            perm = torch.from_numpy(perm_np).to(DEV)
            h.gated_copy(src, dst, perm, gated=True, stamps=True)
            assert h.sync_status() == 0
            assert np.array_equal(dst.cpu().numpy(), oracle.copy_perm(src.cpu().numpy(), perm_np))
            _check_ctrl(h, r)
            n_chunks = (n + 63) // 64
            pub, obs = h.read_latency(n_chunks)
            assert np.all(pub > 0) and np.all(obs >= pub)
        # the ungated control copies the same way and is not a round
        dst2 = torch.zeros_like(src)
        h.gated_copy(src, dst2, perm, gated=False)
        assert h.sync_status() == 0
        assert torch.equal(dst2, dst)
        _check_ctrl(h, 2)


# ------------------------------------------------------------------ edge cases
def test_empty_dispatch_round_then_normal_rounds():
    # T = 0: a round without routed pairs; the plan is empty, nothing is
    # copied or computed, and the next rounds are normal
    H, N, E = 64, 256, 3
    with _handle() as h:
        x0 = torch.zeros(0, H, dtype=torch.bfloat16, device=DEV)
        W = workloads.bf16_normal((E, H, N), 1.0, 61, DEV)
        topk0 = np.zeros((0, 2), np.int32)
        dispatched, offs, out = _dispatch_round(h, x0, topk0, W)
        assert h.sync_status() == 0
        counts, dst, src, pad, blk, m_pad = h.read_plan(0, 2, E)
        assert m_pad == 0 and np.array_equal(counts, np.zeros(E, np.int32))
        assert np.array_equal(offs.cpu().numpy(), np.zeros(E + 1, np.int32))
        _check_ctrl(h, 1)
        for r in (2, 3):
            topk_np = workloads.uniform_topk(90, 2, E, r)
            x = workloads.bf16_normal((90, H), 1.0, 60 + r, DEV)
            dispatched, offs, out = _dispatch_round(h, x, topk_np, W)
            assert h.sync_status() == 0
            _check_dispatch(h, x, topk_np, W, dispatched, offs, out, r)


def test_combine_after_empty_dispatch_is_a_no_op():
    H, N, E = 64, 256, 3
    with _handle() as h:
        _dispatch_round(h, torch.zeros(0, H, dtype=torch.bfloat16, device=DEV), np.zeros((0, 2), np.int32),
                        workloads.bf16_normal((E, H, N), 1.0, 62, DEV))
        y = workloads.bf16_normal((256, N), 1.0, 63, DEV)
        staging = torch.full((1, N), 5.0, dtype=torch.bfloat16, device=DEV)
        combined = torch.full((1, N), 5.0, dtype=torch.bfloat16, device=DEV)
        h.combine(y, torch.ones(1, dtype=torch.float32, device=DEV), staging, combined)
        assert h.sync_status() == 0
        assert torch.all(combined == 5.0) and torch.all(staging == 5.0)
        _check_ctrl(h, 1)


def test_gated_copy_rejects_zero_rows():
    with _handle(max_rows=64) as h:
        src = torch.zeros(1, 64, dtype=torch.uint8, device=DEV)
        perm = torch.zeros(1, dtype=torch.int32, device=DEV)
        with pytest.raises(tovl.TovlError):
            h.gated_copy(src[:0], src[:0], perm[:0])
        assert h.sync_status() == 0


@pytest.mark.parametrize("pairs", [1, 0])
def test_gather_gemm_widest_rows(pairs):
    # K = 32768, the largest supported row (one 64 KB row per producer pass)
    cfg = workloads.GatherCfg("widest", 2, 64, 32768, 256, rounds=1)
    with _handle(producer_ctas=4, k_slices=1) as h:
        h.set_option(tovl.OPT_PAIRS, pairs)
        X, W, gathered, out = _gather_round(h, cfg, 71)
        assert h.sync_status() == 0
        G = oracle.gather([bits(X[s]) for s in range(cfg.shards)])
        assert np.array_equal(bits(gathered), G)
        assert_close(out, oracle.matmul_f32(G, bits(W)), "K = 32768")
        _check_ctrl(h, 1)


def test_gather_gemm_most_shards():
    # 64 shards (the most a call takes) of 24 rows each: chunks span shards
    cfg = workloads.GatherCfg("many shards", 64, 24, 128, 256, rounds=1)
    with _handle(producer_ctas=8, k_slices=2) as h:
        X, W, gathered, out = _gather_round(h, cfg, 72)
        assert h.sync_status() == 0
        G = oracle.gather([bits(X[s]) for s in range(cfg.shards)])
        assert np.array_equal(bits(gathered), G)
        assert_close(out, oracle.matmul_f32(G, bits(W)), "64 shards")
        _check_ctrl(h, 1)


def test_dispatch_most_experts():
    # 512 experts (the most a call takes), most of them empty or with one row
    H, N, E = 64, 256, 512
    with _handle(max_experts=E, max_rows=1 << 17) as h:
        for r in (1, 2):
            topk_np = workloads.uniform_topk(300, 2, E, 80 + r)
            x = workloads.bf16_normal((300, H), 1.0, 82 + r, DEV)
            W = workloads.bf16_normal((E, H, N), 1.0, 84 + r, DEV)
            dispatched, offs, out = _dispatch_round(h, x, topk_np, W)
            assert h.sync_status() == 0
            _check_dispatch(h, x, topk_np, W, dispatched, offs, out, r)


def test_dispatch_pair_tiles_phantom_half_at_buffer_end():
    # 128-row segments on CTA pairs (the default): two experts of one row
    # each fill the whole buffer (rows = m_pad = 256), so every pair tile is
    # one block and a phantom half, the last one past the end of the buffer;
    # then experts of 3, 1 and 2 blocks (odd and even block counts)
    H, N = 128, 256
    with _handle(k_slices=2) as h:
        assert h.get_option(tovl.OPT_EMBEDDED) == 1 and h.get_option(tovl.OPT_DISPATCH_ALIGN) == 128
        cases = [np.array([[0], [1]], dtype=np.int32),
                 np.concatenate([np.zeros((300, 1)), np.ones((100, 1)), np.full((200, 1), 2)]).astype(np.int32)]
        for r, topk_np in enumerate(cases, start=1):
            T, k = topk_np.shape
            E = int(topk_np.max()) + 1
            assert r > 1 or tovl.dispatch_rows(T, k, E) == 256
            x = workloads.bf16_normal((T, H), 1 / math.sqrt(H), 990 + r, DEV)
            W = workloads.bf16_normal((E, H, N), 1 / math.sqrt(H), 995 + r, DEV)
            dispatched, offs, out = _dispatch_round(h, x, topk_np, W)
            assert h.sync_status() == 0
            _check_dispatch(h, x, topk_np, W, dispatched, offs, out, r)


@pytest.mark.parametrize("routing", list(ROUTINGS))
@pytest.mark.parametrize("H,N,KS", [(192, 512, 2), (320, 1536, 3), (1024, 1024, 1)])
@pytest.mark.parametrize("wide", [1, 0])
def test_dispatch_wide_pair_tiles(routing, H, N, KS, wide):
    # option 23: CTA-pair tiles on the plan's pair table 512 columns wide (one
    # 512-column accumulator, the weights as one 4-D box per k-block) or 256
    # wide; N = 1536 gives three 512-column blocks, H = 320 five k-blocks
    # over three K-slices; every routing has phantom halves
    with _handle(k_slices=KS) as h:
        h.set_option(tovl.OPT_WIDE_TILES, wide)
        assert h.get_option(tovl.OPT_WIDE_TILES) == wide
        for r in range(1, 4):
            topk_np, E = ROUTINGS[routing](workloads.round_seed(6, r))
            T = topk_np.shape[0]
            x = workloads.bf16_normal((T, H), 1 / math.sqrt(H), 400 + r, DEV)
            W = workloads.bf16_normal((E, H, N), 1 / math.sqrt(H), 410 + r, DEV)
            dispatched, offs, out = _dispatch_round(h, x, topk_np, W)
            assert h.sync_status() == 0
            _check_dispatch(h, x, topk_np, W, dispatched, offs, out, r)


@pytest.mark.parametrize("routing", list(ROUTINGS))
@pytest.mark.parametrize("wide", [1, 0])
def test_dispatch_wide_pair_tiles_on_256_row_segments(routing, wide):
    # option 17 = 256 with embedded producers: 256-row segments, CTA-pair
    # tiles 512 (wide) or 256 columns wide, N = 1024
    H, N, align = 256, 1024, 256
    with _handle(k_slices=2) as h:
        h.set_option(tovl.OPT_DISPATCH_ALIGN, align)
        h.set_option(tovl.OPT_WIDE_TILES, wide)
        for r in range(1, 3):
            topk_np, E = ROUTINGS[routing](workloads.round_seed(8, r))
            T, k = topk_np.shape
            x = workloads.bf16_normal((T, H), 1 / math.sqrt(H), 430 + r, DEV)
            W = workloads.bf16_normal((E, H, N), 1 / math.sqrt(H), 440 + r, DEV)
            rows = tovl.dispatch_rows_aligned(T, k, E, align)
            dispatched = torch.full((rows, H), 3.0, dtype=torch.bfloat16, device=DEV)
            offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
            out = torch.empty(rows, N, dtype=torch.bfloat16, device=DEV)
            h.dispatch_grouped_gemm(x, torch.from_numpy(topk_np).to(DEV), W, dispatched, offs, out)
            assert h.sync_status() == 0
            p = oracle.dispatch_plan(topk_np, E, block_rows=align)
            counts, dst, src, pad, blk, m_pad = h.read_plan(T, k, E)
            assert m_pad == p.m_pad
            assert np.array_equal(dst, p.dst)
            D = oracle.dispatch(bits(x), p.dst, k, p.m_pad)
            assert np.array_equal(bits(dispatched[:m_pad]), D), "dispatched buffer"
            assert_close(out[:m_pad], oracle.grouped_matmul_f32(D, bits(W), p.off), f"256-row segments, wide {wide}")
            _check_ctrl(h, r)


def test_option_ranges_are_checked():
    # each documented option value round-trips; a value outside the
    # documented range is rejected with TOVL_ERR_INVALID and leaves the
    # option as it was
    cases = {tovl.OPT_PDL: ([0, 1], [2, -1]), tovl.OPT_ROLE_SWITCH: ([0, 1, 2], [3, -1]),
             tovl.OPT_DISPATCH_ALIGN: ([256, 128], [64, 192, 512]), tovl.OPT_EMBEDDED: ([0, 2, 1], [3, -1]),
             tovl.OPT_RS_EPILOGUE: ([1, 0], [2, -1]), tovl.OPT_L2_HINTS: ([0, 63, -1], [64, -2]),
             tovl.OPT_WIDE_TILES: ([0, 1], [2, -1])}
    with _handle() as h:
        for opt, (good, bad) in cases.items():
            for v in good:
                h.set_option(opt, v)
                assert h.get_option(opt) == v
            for v in bad:
                with pytest.raises(tovl.TovlError) as e:
                    h.set_option(opt, v)
                assert e.value.code == tovl.TOVL_ERR_INVALID
                assert h.get_option(opt) == good[-1]


def test_dispatch_wide_pair_tiles_phantom_half_at_buffer_end():
    # 512-column pair tiles whose second block is a phantom past the end of
    # the buffer (two one-row experts fill rows = m_pad = 256)
    H, N = 128, 512
    with _handle(k_slices=2) as h:
        assert h.get_option(tovl.OPT_WIDE_TILES) == 1
        topk_np = np.array([[0], [1]], dtype=np.int32)
        T, k = topk_np.shape
        assert tovl.dispatch_rows(T, k, 2) == 256
        x = workloads.bf16_normal((T, H), 1 / math.sqrt(H), 420, DEV)
        W = workloads.bf16_normal((2, H, N), 1 / math.sqrt(H), 421, DEV)
        dispatched, offs, out = _dispatch_round(h, x, topk_np, W)
        assert h.sync_status() == 0
        _check_dispatch(h, x, topk_np, W, dispatched, offs, out, 1)


@pytest.mark.parametrize("routing", list(ROUTINGS))
@pytest.mark.parametrize("align,pairs", [(128, 1), (256, 1), (128, 0)])
def test_dispatch_embedded_producers(routing, align, pairs):
    # option 18: no producer CTAs; the consumer CTAs' spare warps copy the
    # rows; the same plan, buffers and counters as with producer CTAs.  With
    # CTA pairs off the single-CTA kernel runs (its prologue barrier counts
    # warps 0-10 and the stage waiter, not the copy warps)
    H, N = 192, 512
    with _handle(k_slices=2) as h:
        h.set_option(tovl.OPT_PAIRS, pairs)
        h.set_option(tovl.OPT_DISPATCH_ALIGN, align)
        h.set_option(tovl.OPT_EMBEDDED, 1)
        assert h.get_option(tovl.OPT_EMBEDDED) == 1
        for r in range(1, 4):
            topk_np, E = ROUTINGS[routing](workloads.round_seed(4, r))
            T, k = topk_np.shape
            x = workloads.bf16_normal((T, H), 1 / math.sqrt(H), 960 + r, DEV)
            W = workloads.bf16_normal((E, H, N), 1 / math.sqrt(H), 970 + r, DEV)
            rows = tovl.dispatch_rows_aligned(T, k, E, align)
            dispatched = torch.full((rows, H), 3.0, dtype=torch.bfloat16, device=DEV)
            offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
            out = torch.empty(rows, N, dtype=torch.bfloat16, device=DEV)
            h.dispatch_grouped_gemm(x, torch.from_numpy(topk_np).to(DEV), W, dispatched, offs, out)
            assert h.sync_status() == 0
            assert h.get_option(tovl.OPT_PRODUCERS) == 0
            p = oracle.dispatch_plan(topk_np, E, block_rows=align)
            counts, dst, src, pad, blk, m_pad = h.read_plan(T, k, E)
            assert m_pad == p.m_pad
            assert np.array_equal(offs.cpu().numpy(), p.off)
            assert np.array_equal(dst, p.dst)
            assert np.array_equal(src, p.src)
            D = oracle.dispatch(bits(x), p.dst, k, p.m_pad)
            assert np.array_equal(bits(dispatched[:m_pad]), D), "dispatched buffer"
            assert_close(out[:m_pad], oracle.grouped_matmul_f32(D, bits(W), p.off), "embedded producers")
            _check_ctrl(h, r)


@pytest.mark.parametrize("mask", [0, 1, 2, 4, 8, 16, 32, 63])
def test_l2_eviction_hints_leave_results_unchanged(mask):
    # option 20 only changes L2 eviction priorities: the gather + GEMM and the
    # dispatch + grouped GEMM agree with the oracle under every hint bit
    cfg = workloads.GatherCfg("hints", 3, 200, 320, 512, rounds=2)
    with _handle(producer_ctas=6, k_slices=2) as h:
        h.set_option(tovl.OPT_L2_HINTS, mask)
        assert h.get_option(tovl.OPT_L2_HINTS) == mask
        X, W, gathered, out = _gather_round(h, cfg, 40 + mask)
        assert h.sync_status() == 0
        G = oracle.gather([bits(X[s]) for s in range(cfg.shards)])
        assert np.array_equal(bits(gathered), G)
        assert_close(out, oracle.matmul_f32(G, bits(W)), f"gather, hints {mask}")
        topk_np, E = ROUTINGS["zipf"](workloads.round_seed(9, mask))
        T = topk_np.shape[0]
        x = workloads.bf16_normal((T, 192), 1 / math.sqrt(192), 50 + mask, DEV)
        Wd = workloads.bf16_normal((E, 192, 256), 1 / math.sqrt(192), 60 + mask, DEV)
        dispatched, offs, outd = _dispatch_round(h, x, topk_np, Wd)
        assert h.sync_status() == 0
        _check_dispatch(h, x, topk_np, Wd, dispatched, offs, outd, 2)
