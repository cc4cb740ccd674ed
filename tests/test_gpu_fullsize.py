"""GPU parity at the benchmarked sizes, in the launch configurations bench.py
times (the same handle settings and automatic CTA splits), over each
configuration's stated round count with sequences never reset.

Buffers, routing plans and control-plane state are compared whole and bit for
bit with the oracle.  GEMM outputs are compared whole in the first and last
rounds of the TP workload and in the first round of every dispatch
configuration (and its last round in the default one); in the other rounds on
seeded samples of rows that the oracle computes one row at a time (first and
last rows, shard and block boundaries, and random rows).  Tolerance:
|gpu - oracle| <= 2e-2 + 1e-2 |oracle| elementwise.
"""
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


def _rows(n: int, must, count: int, seed: int) -> np.ndarray:
    """Sorted unique sample of [0, n): the listed rows plus `count` random ones."""
    rng = np.random.default_rng(seed)
    picked = set(int(r) for r in must if 0 <= r < n)
    picked.update(int(r) for r in rng.choice(n, size=min(count, n), replace=False))
    return np.array(sorted(picked), dtype=np.int64)


def _check_ctrl(h, R):
    slots, cnts, rb, seq = h.read_ctrl()
    o_slots, o_cnts, o_rb = oracle.ctrl_state(R, slots.size, rb.size)
    assert seq == R
    assert np.array_equal(slots, o_slots), "slots"
    assert np.array_equal(cnts, o_cnts), "chunk counters"
    assert np.array_equal(rb, o_rb), "row-block counters"


def _on(t: torch.Tensor, rows: np.ndarray) -> torch.Tensor:
    return t[torch.from_numpy(rows).to(t.device)]


def test_tp_gather_gemm_full_size():
    # 4 shards x 768 rows, K = N = 4096, the configuration's 20 rounds with
    # new inputs every round and sequences never reset: the handle bench.py
    # times the TP step with (automatic producer / consumer split, CTA pairs,
    # 4 K-slices)
    cfg = workloads.TP
    R = cfg.rows_per_shard
    must = [0, 127, 128, 255, 256, R - 1, R, 2 * R - 1, 2 * R, cfg.M - 129, cfg.M - 128, cfg.M - 1]
    with tovl.Handle(0, max_rows=1 << 14, k_slices=4) as h:
        for r in range(1, cfg.rounds + 1):
            X, W = workloads.gather_inputs(cfg, workloads.round_seed(cfg.seed, r), DEV)
            gathered = torch.full((cfg.M, cfg.K), 3.0, dtype=torch.bfloat16, device=DEV)
            out = torch.empty(cfg.M, cfg.N, dtype=torch.bfloat16, device=DEV)
            h.gather_gemm(X, W, gathered, out)
            assert h.sync_status() == 0
            G = oracle.gather([bits(X[s]) for s in range(cfg.shards)])
            assert np.array_equal(bits(gathered), G), f"gathered buffer, round {r}"
            if r in (1, cfg.rounds):
                # the whole output: every tile of the three-wave pair schedule
                assert_close(out, oracle.matmul_f32(G, bits(W)), f"TP output, round {r}")
            else:
                rows = _rows(cfg.M, must, 6, r)
                assert_close(_on(out, rows), oracle.matmul_rows_f32(G, bits(W), rows), f"TP output rows, round {r}")
            _check_ctrl(h, r)


def _dispatch_full_round(h, cfg, align, r, dispatched, offs, out, whole=False):
    x, topk_np, W = workloads.dispatch_inputs(cfg, r - 1, DEV)
    h.dispatch_grouped_gemm(x, torch.from_numpy(topk_np).to(DEV), W, dispatched, offs, out)
    assert h.sync_status() == 0
    p = oracle.dispatch_plan(topk_np, cfg.E, block_rows=align)
    counts, dst, src, pad, blk, m_pad = h.read_plan(cfg.T, cfg.k, cfg.E)
    assert m_pad == p.m_pad
    assert np.array_equal(counts, p.counts)
    assert np.array_equal(offs.cpu().numpy(), p.off)
    assert np.array_equal(dst, p.dst)
    assert np.array_equal(src, p.src)
    # per 128-row block: padding = rows without a source, expert = segment
    real = (p.src >= 0).reshape(-1, 128).sum(axis=1)
    assert np.array_equal(pad, 128 - real)
    assert np.array_equal(blk, np.searchsorted(p.off, np.arange(0, m_pad, 128), side="right") - 1)
    D = oracle.dispatch(bits(x), p.dst, cfg.k, p.m_pad)
    assert np.array_equal(bits(dispatched[:m_pad]), D), f"dispatched buffer, round {r}"
    if whole:
        # every output row of every expert segment (padding rows included)
        assert_close(out[:m_pad], oracle.grouped_matmul_f32(D, bits(W), p.off), f"grouped GEMM, round {r}")
    else:
        # sampled real rows of every expert (its first and last row among them)
        for e in range(cfg.E):
            lo, n_e = int(p.off[e]), int(p.counts[e])
            if n_e == 0:
                continue
            rows = _rows(n_e, [0, n_e - 1], 2, e) + lo
            assert_close(_on(out, rows), oracle.matmul_rows_f32(D, bits(W[e]), rows), f"expert {e}, round {r}")
    # padding rows of the output are exact zeros
    pad_rows = np.nonzero(p.src < 0)[0]
    if pad_rows.size:
        assert torch.count_nonzero(_on(out, pad_rows)) == 0
    _check_ctrl(h, r)


@pytest.mark.parametrize("name,align", [("DISPATCH", 128), ("DISPATCH", 256), ("SKEWED", 128), ("SKEWED", 256)])
@pytest.mark.parametrize("embedded", [1, 0])
def test_dispatch_grouped_gemm_full_size(name, align, embedded):
    # uniform top-2 of 8 (T=4096, H=4096) and Zipf(1.2) top-4 of 32 (T=8192,
    # H=7168), N=2048; 128- and 256-row segments, with embedded producers
    # (the default) and with producer CTAs: the handles bench.py's dispatch
    # lines use.  The configuration's ten rounds, a new routing each (the
    # padding rows move between rounds and must be zero again), sequences
    # never reset.
    cfg = getattr(workloads, name)
    rows_cap = tovl.dispatch_rows_aligned(cfg.T, cfg.k, cfg.E, align)
    with tovl.Handle(0, max_rows=rows_cap, max_pairs=cfg.T * cfg.k, max_experts=cfg.E, k_slices=4) as h:
        h.set_option(tovl.OPT_DISPATCH_ALIGN, align)
        h.set_option(tovl.OPT_EMBEDDED, embedded)   # 1: the default, copy warps in the consumer CTAs
        dispatched = torch.full((rows_cap, cfg.H), 3.0, dtype=torch.bfloat16, device=DEV)
        offs = torch.empty(cfg.E + 1, dtype=torch.int32, device=DEV)
        out = torch.empty(rows_cap, cfg.N, dtype=torch.bfloat16, device=DEV)
        default = align == 128 and embedded == 1
        for r in range(1, cfg.rounds + 1):
            whole = r == 1 or (default and r == cfg.rounds)
            _dispatch_full_round(h, cfg, align, r, dispatched, offs, out, whole=whole)


@pytest.mark.parametrize("name", ["DISPATCH", "SKEWED"])
def test_combine_full_size(name):
    # combine after the uniform top-2 and the Zipf top-4 dispatch, on their
    # expert outputs, with the handle and CTA split bench.py's combine lines use
    cfg = getattr(workloads, name)
    x, topk_np, W = workloads.dispatch_inputs(cfg, 0, DEV)
    rows_cap = tovl.dispatch_rows(cfg.T, cfg.k, cfg.E)
    with tovl.Handle(0, max_rows=rows_cap, max_pairs=cfg.T * cfg.k, max_experts=cfg.E, k_slices=4) as h:
        dispatched = torch.zeros(rows_cap, cfg.H, dtype=torch.bfloat16, device=DEV)
        offs = torch.empty(cfg.E + 1, dtype=torch.int32, device=DEV)
        y = torch.empty(rows_cap, cfg.N, dtype=torch.bfloat16, device=DEV)
        h.dispatch_grouped_gemm(x, torch.from_numpy(topk_np).to(DEV), W, dispatched, offs, y)
        w_np = workloads.gate_weights(cfg.T, cfg.k, 0)
        staging = torch.full((cfg.T * cfg.k, cfg.N), 5.0, dtype=torch.bfloat16, device=DEV)
        combined = torch.full((cfg.T, cfg.N), 5.0, dtype=torch.bfloat16, device=DEV)
        h.combine(y, torch.from_numpy(w_np).to(DEV), staging, combined)
        assert h.sync_status() == 0
        S, C = oracle.combine(bits(y), oracle.dispatch_plan(topk_np, cfg.E).dst, w_np)
        assert np.array_equal(bits(staging), S), "staging"
        assert np.array_equal(bits(combined), C), "combined"
        _check_ctrl(h, 2)


def test_gemm_reduce_scatter_full_size():
    # the TP shape split four ways along K (K/S = 1024), with the handle and
    # automatic split of bench.py's reduce-scatter line
    cfg = workloads.TP
    S, M, K, N = cfg.shards, cfg.M, cfg.K, cfg.N
    Ks = K // S
    X = workloads.bf16_normal((S, M, Ks), 1 / K ** 0.5, 0, DEV)
    W = workloads.bf16_normal((S, Ks, N), 1 / K ** 0.5, 1, DEV)
    partials = torch.full((S, M, N), 3.0, dtype=torch.bfloat16, device=DEV)
    out = torch.full((M, N), 3.0, dtype=torch.bfloat16, device=DEV)
    with tovl.Handle(0, max_rows=1 << 14, k_slices=4) as h:
        h.gemm_reduce_scatter(X, W, partials, out)
        assert h.sync_status() == 0
        rows = _rows(M, [0, 255, 256, M - 1], 24, 5)
        Pr = np.stack([oracle.f32_to_bf16(oracle.matmul_rows_f32(bits(X[s]), bits(W[s]), rows)) for s in range(S)])
        for s in range(S):
            assert_close(_on(partials[s], rows), oracle.bf16_to_f32(Pr[s]), f"partial {s}")
        assert_close(_on(out, rows), oracle.bf16_to_f32(oracle.reduce_partials(Pr)), "reduced rows")
        _check_ctrl(h, 1)


@pytest.mark.parametrize("row_bytes,mode", [(256, 0), (1024, 0), (8192, 0), (16384, 0), (256, 1), (16384, 1),
                                            (8192, 2)])
def test_gated_copy_full_size(row_bytes, mode):
    # 2^20 permuted rows (256 B - 16 KB, up to 16 GiB each way), the copy
    # line's handle in the vector (0), bulk (1) and default automatic (2)
    # modes, two rounds
    cfg = workloads.COPY
    n, rb = cfg.n_rows, row_bytes
    perm_np = workloads.permutation(n, cfg.seed)
    perm = torch.from_numpy(perm_np).to(DEV)
    rows = _rows(n, [0, n - 1], 2048, 7)
    dests = perm_np[rows].astype(np.int64)
    rank = np.argsort(np.argsort(dests)).astype(np.int32)
    with tovl.Handle(0, max_rows=n, copy_mode=mode) as h:
        src = torch.empty(n, rb, dtype=torch.uint8, device=DEV)
        dst = torch.zeros_like(src)
        for r in (1, 2):
            src.random_(0, 256)
            h.gated_copy(src, dst, perm, gated=True)
            assert h.sync_status() == 0
            # the sample of source rows as a smaller copy for the oracle: row j
            # of the sample goes to the rank of its destination in the sample
            want = oracle.copy_perm(_on(src, rows).cpu().numpy(), rank)
            got = _on(dst, np.sort(dests)).cpu().numpy()
            assert np.array_equal(got, want), f"sampled destination rows, round {r}"
            _check_ctrl(h, r)
        del src, dst
        torch.cuda.empty_cache()


def test_gated_copy_thousand_rounds():
    # the sweep's 1000 rounds of monotonic sequence numbers (256 B rows):
    # the control plane's closed form after every 100th round and the data of
    # the last round
    cfg = workloads.COPY
    n, rb = cfg.n_rows, 256
    perm_np = workloads.permutation(n, cfg.seed)
    perm = torch.from_numpy(perm_np).to(DEV)
    with tovl.Handle(0, max_rows=n) as h:
        src = workloads.random_bytes(n, rb, 3, DEV)
        dst = torch.zeros_like(src)
        for r in range(1, cfg.rounds + 1):
            h.gated_copy(src, dst, perm, gated=True)
            if r % 100 == 0:
                assert h.sync_status() == 0
                _check_ctrl(h, r)
        assert np.array_equal(dst.cpu().numpy(), oracle.copy_perm(src.cpu().numpy(), perm_np))
