"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: a library
routine (numpy / torch), a hand-worked case, brute force over every routing
of a tiny problem, or an independent simulation of the sync protocol.  A
plausible slip in the oracle (dropped term, wrong index, transposed operand,
wrong rounding, wrong accumulate precision) fails at least one of them.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
import workloads


def _bf16_bits_from_f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def _f64_from_bits(h):
    return torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


# ------------------------------------------------------------------ bf16
def test_bf16_widening_matches_torch():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 1 << 16, size=100000, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]          # finite values
    ours = oracle.bf16_to_f32(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))


def test_bf16_rounding_hand_cases():
    # 1 + 2^-8 is a tie between 0x3F80 and 0x3F81 -> even 0x3F80;
    # 1 + 3*2^-8 is a tie between 0x3F81 and 0x3F82 -> even 0x3F82;
    # 1 + 2^-8 + 2^-20 is above the tie -> 0x3F81.
    vals = np.array([1.0, 1 + 2**-8, 1 + 3 * 2**-8, 1 + 2**-8 + 2**-20, -2.0, 0.0, np.inf],
                    np.float32)
    assert list(oracle.f32_to_bf16(vals)) == [0x3F80, 0x3F80, 0x3F82, 0x3F81, 0xC000, 0x0000, 0x7F80]
    nan = oracle.f32_to_bf16(np.array([np.nan], np.float32))[0]
    assert (nan & 0x7F80) == 0x7F80 and (nan & 0x007F) != 0


def test_bf16_rounding_matches_torch_rne():
    rng = np.random.default_rng(2)
    f = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * 10.0,
        rng.integers(0, 1 << 32, size=200000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])
    f = f[np.isfinite(f)]
    ours = oracle.f32_to_bf16(f)
    ref = _bf16_bits_from_f32(f)
    assert np.array_equal(ours, ref)


# ------------------------------------------------------------------ matmul
def test_matmul_hand_case():
    A = _bf16_bits_from_f32(np.array([[1, 2], [3, 4]], np.float32))
    W = _bf16_bits_from_f32(np.array([[5, 6], [7, 8]], np.float32))
    assert np.array_equal(oracle.matmul_f32(A, W), np.array([[19, 22], [43, 50]], np.float32))


@pytest.mark.parametrize("M,N,K", [(5, 3, 7), (17, 33, 64), (64, 40, 300)])
def test_matmul_within_fp32_bound_of_float64(M, N, K):
    rng = np.random.default_rng(M * 1000 + N)
    A = _bf16_bits_from_f32(rng.standard_normal((M, K)))
    W = _bf16_bits_from_f32(rng.standard_normal((K, N)))
    a, w = _f64_from_bits(A), _f64_from_bits(W)
    ref = a @ w                                 # float64 textbook product
    bound = K * 2.0**-24 * (np.abs(a) @ np.abs(w)) + 1e-30
    got = oracle.matmul_f32(A, W).astype(np.float64)
    assert np.all(np.abs(got - ref) <= bound)
    # a transposed or mis-indexed operand is far outside the bound
    assert np.max(np.abs(got - ref)) < 1e-3 * np.max(np.abs(ref))


def test_matmul_identity_returns_input_exactly():
    rng = np.random.default_rng(3)
    A = _bf16_bits_from_f32(rng.standard_normal((9, 32)))
    I = _bf16_bits_from_f32(np.eye(32, dtype=np.float32))
    assert np.array_equal(oracle.matmul_f32(A, I), oracle.bf16_to_f32(A))


def test_matmul_accumulates_in_fp32_in_ascending_k():
    # 2^24 + 1 rounds to 2^24 in fp32 (tie to even); minus 2^24 gives 0.
    # A float64 (or reordered) sum would give 1.
    A = _bf16_bits_from_f32(np.array([[2.0**24, 1.0, -(2.0**24)]], np.float32))
    W = _bf16_bits_from_f32(np.ones((3, 1), np.float32))
    assert oracle.matmul_f32(A, W)[0, 0] == 0.0
    A2 = _bf16_bits_from_f32(np.array([[1.0, 2.0**24, -(2.0**24)]], np.float32))
    assert oracle.matmul_f32(A2, W)[0, 0] == 0.0   # 1 + 2^24 also rounds to 2^24
    A3 = _bf16_bits_from_f32(np.array([[2.0**24, -(2.0**24), 1.0]], np.float32))
    assert oracle.matmul_f32(A3, W)[0, 0] == 1.0


def test_matmul_rows_matches_full():
    rng = np.random.default_rng(4)
    A = _bf16_bits_from_f32(rng.standard_normal((40, 96)))
    W = _bf16_bits_from_f32(rng.standard_normal((96, 24)))
    rows = np.array([0, 39, 7, 7, 20])
    assert np.array_equal(oracle.matmul_rows_f32(A, W, rows), oracle.matmul_f32(A, W)[rows])


# ------------------------------------------------------------------ gather / copy
def test_gather_is_concatenation():
    X, _ = workloads.gather_inputs(workloads.TINY, seed=0)
    shards = [workloads.bf16_bits(X[s]) for s in range(X.shape[0])]
    G = oracle.gather(shards)
    assert np.array_equal(G, np.concatenate(shards, axis=0))


def test_gather_expected_matches_bincount():
    for n in [1, 63, 64, 65, 256, 3072, 1000]:
        exp = oracle.gather_expected(n)
        ref = np.bincount(np.arange(n) // 64, minlength=(n + 63) // 64)
        assert np.array_equal(exp, ref)


def test_copy_perm_matches_numpy_scatter():
    perm = workloads.permutation(1000, 5)
    src = workloads.random_bytes(1000, 48, 5).numpy()
    ref = np.empty_like(src)
    ref[perm] = src
    assert np.array_equal(oracle.copy_perm(src, perm), ref)
    assert np.array_equal(oracle.perm_expected(perm), np.bincount(perm // 64, minlength=16))


# ------------------------------------------------------------------ dispatch plan
def test_dispatch_plan_hand_worked():
    # T=4, k=2, E=3, blocks of 2 rows.  Counts: e0 <- (0,0),(2,0),(3,1);
    # e1 <- (1,1),(2,1); e2 <- (0,1),(1,0),(3,0).  Padded sizes 4, 2, 4.
    topk = np.array([[0, 2], [2, 1], [0, 1], [2, 0]], np.int32)
    p = oracle.dispatch_plan(topk, E=3, block_rows=2)
    assert list(p.counts) == [3, 2, 3]
    assert list(p.off) == [0, 4, 6, 10]
    assert list(p.dst) == [0, 6, 7, 4, 1, 5, 8, 2]
    assert list(p.src) == [0, 2, 3, -1, 1, 2, 0, 1, 3, -1]
    assert list(p.pad) == [0, 1, 0, 0, 1]
    assert list(p.blk_e) == [0, 0, 1, 2, 2]


def _plan_by_sorting(topk, E, B):
    """Independent formulation: a stable sort of the flattened expert ids."""
    ids = topk.reshape(-1)
    counts = np.bincount(ids, minlength=E)
    padded = (counts + B - 1) // B * B
    off = np.concatenate([[0], np.cumsum(padded)])
    order = np.argsort(ids, kind="stable")
    first = np.concatenate([[0], np.cumsum(counts)])[:-1]
    dst = np.empty(ids.size, np.int64)
    for pos, i in enumerate(order):
        e = ids[i]
        dst[i] = off[e] + (pos - first[e])
    return counts, off, dst


def _check_plan(topk, E, B):
    p = oracle.dispatch_plan(topk, E=E, block_rows=B)
    counts, off, dst = _plan_by_sorting(topk, E, B)
    assert np.array_equal(p.counts, counts)
    assert np.array_equal(p.off, off)
    assert np.array_equal(p.dst, dst)
    T, k = topk.shape
    src = np.full(off[-1], -1)
    src[dst] = np.repeat(np.arange(T), k)
    assert np.array_equal(p.src, src)
    real = (src >= 0).reshape(-1, B).sum(axis=1) if off[-1] else np.zeros(0)
    assert np.array_equal(p.pad, B - real)
    assert int(p.pad.sum()) == off[-1] - T * k
    owner = np.searchsorted(off, np.arange(0, off[-1], B), side="right") - 1
    assert np.array_equal(p.blk_e, owner)


def test_dispatch_plan_brute_force_all_routings():
    # every routing of T tokens to k distinct experts out of E, T<=3, E<=3, k<=2
    for T, E, k, B in [(1, 1, 1, 2), (2, 2, 1, 2), (3, 3, 2, 2), (2, 3, 2, 1), (3, 2, 2, 4)]:
        choices = list(itertools.permutations(range(E), k))
        for combo in itertools.product(choices, repeat=T):
            _check_plan(np.array(combo, np.int32).reshape(T, k), E, B)


@pytest.mark.parametrize("routing", ["uniform", "zipf", "one", "empty_expert"])
def test_dispatch_plan_matches_sort_on_workloads(routing):
    if routing == "uniform":
        topk, E = workloads.uniform_topk(4096, 2, 8, 0), 8
    elif routing == "zipf":
        topk, E = workloads.zipf_topk(8192, 4, 32, 1.2, 0), 32
    elif routing == "one":
        topk, E = workloads.all_to_one_topk(300, 4, 2), 4
    else:
        topk, E = workloads.uniform_topk(500, 2, 5, 1), 7      # experts 5, 6 unused
    _check_plan(topk, E, 128)


def test_dispatch_plan_rejects_bad_ids():
    with pytest.raises(ValueError):
        oracle.dispatch_plan(np.array([[0, 3]], np.int32), E=3)
    with pytest.raises(ValueError):
        oracle.dispatch_plan(np.array([[0, -1]], np.int32), E=3)


def test_dispatch_rows_and_zero_padding():
    rng = np.random.default_rng(6)
    x = rng.integers(1, 1 << 15, size=(50, 16), dtype=np.uint16)   # no zero rows
    topk = workloads.uniform_topk(50, 2, 4, 6)
    p = oracle.dispatch_plan(topk, E=4)
    D = oracle.dispatch(x, p.dst, 2, p.m_pad)
    for t in range(50):
        for j in range(2):
            assert np.array_equal(D[p.dst[t * 2 + j]], x[t])
    assert np.all(D[p.src < 0] == 0)
    assert np.all(np.any(D[p.src >= 0] != 0, axis=1))


def test_dispatch_single_expert_reduces_to_gather():
    rng = np.random.default_rng(7)
    x = rng.integers(0, 1 << 16, size=(256, 8), dtype=np.uint16)
    p = oracle.dispatch_plan(np.zeros((256, 1), np.int32), E=1)
    assert p.m_pad == 256 and np.array_equal(oracle.dispatch(x, p.dst, 1, p.m_pad), x)


def test_grouped_matmul_per_segment_and_padding_zero():
    rng = np.random.default_rng(8)
    topk = workloads.uniform_topk(200, 2, 3, 8)
    p = oracle.dispatch_plan(topk, E=3)
    x = _bf16_bits_from_f32(rng.standard_normal((200, 64)))
    W = _bf16_bits_from_f32(rng.standard_normal((3, 64, 16)))
    D = oracle.dispatch(x, p.dst, 2, p.m_pad)
    O = oracle.grouped_matmul_f32(D, W, p.off)
    d, w = _f64_from_bits(D), _f64_from_bits(W)
    for e in range(3):
        r0, r1 = p.off[e], p.off[e + 1]
        ref = d[r0:r1] @ w[e]
        bound = 64 * 2.0**-24 * (np.abs(d[r0:r1]) @ np.abs(w[e]))
        assert np.all(np.abs(O[r0:r1] - ref) <= bound + 1e-30)
    assert np.all(O[p.src < 0] == 0.0)


def test_gather_single_shard_gemm_is_plain_gemm():
    rng = np.random.default_rng(9)
    X = _bf16_bits_from_f32(rng.standard_normal((64, 32)))
    W = _bf16_bits_from_f32(rng.standard_normal((32, 16)))
    G = oracle.gather([X])
    assert np.array_equal(oracle.matmul_f32(G, W), oracle.matmul_f32(X, W))


# ------------------------------------------------------------------ protocol closed form
def _simulate_protocol(rounds, expected_real, chunk_rows, rng):
    """Independent event simulation of the single-writer protocol.

    Each round, every chunk receives its real arrivals (grouped in random
    batches) and one padding-seed arrival, in random order.  A counter is
    never reset; the arrival whose add brings it to seq*chunk_rows is elected
    and release-stores seq into the chunk's slot."""
    n = len(expected_real)
    cnt = np.zeros(n, np.int64)
    slot = np.zeros(n, np.int64)
    for seq in range(1, rounds + 1):
        for c in range(n):
            arrivals = []
            left = int(expected_real[c])
            while left:
                b = int(rng.integers(1, left + 1))
                arrivals.append(b)
                left -= b
            if chunk_rows - expected_real[c]:
                arrivals.append(chunk_rows - int(expected_real[c]))
            rng.shuffle(arrivals)
            elected = 0
            for a in arrivals:
                old = cnt[c]
                cnt[c] += a
                if old + a == seq * chunk_rows:
                    slot[c] = seq
                    elected += 1
            assert elected == 1                       # exactly one writer per slot per round
            assert slot[c] >= seq                     # round k reads >= k
    return slot, cnt


def test_ctrl_closed_form_matches_protocol_simulation():
    rng = np.random.default_rng(10)
    for n_rows, R in [(256, 3), (200, 5), (3072, 2)]:
        exp = oracle.gather_expected(n_rows)
        slot, cnt = _simulate_protocol(R, exp, 64, rng)
        o_slot, o_cnt, o_rb = oracle.ctrl_state(R, exp.size, 0)
        assert np.array_equal(o_slot, slot) and np.array_equal(o_cnt, cnt)
    # row-block counters: real arrivals + one padding seed reach 128 per round
    p = oracle.dispatch_plan(workloads.zipf_topk(2000, 4, 32, 1.2, 3), E=32)
    slot, cnt = _simulate_protocol(4, 128 - p.pad, 128, rng)
    _, _, o_rb = oracle.ctrl_state(4, 0, p.n_blocks)
    assert np.array_equal(o_rb, cnt)


# ------------------------------------------------------------------ combine
def _plan_dst(topk, E):
    return oracle.dispatch_plan(topk, E).dst.reshape(topk.shape)


@pytest.mark.parametrize("routing", ["uniform", "zipf", "one"])
def test_combine_staging_inverts_dispatch(routing):
    T, k, E, H = 50, 3, 6, 24
    topk = {"uniform": lambda: workloads.uniform_topk(T, k, E, 3),
            "zipf": lambda: workloads.zipf_topk(T, k, E, 1.2, 3),
            "one": lambda: workloads.all_to_one_topk(T, E, 2)}[routing]()
    k = topk.shape[1]
    p = oracle.dispatch_plan(topk, E)
    x = np.random.default_rng(5).integers(0, 1 << 15, size=(T, H), dtype=np.uint16)
    D = oracle.dispatch(x, p.dst, k, p.m_pad)
    S, _ = oracle.combine(D, p.dst, np.ones((T, k), np.float32))
    # every pair's staged row is its own token's row: dispatch followed by the
    # combine scatter is the identity on each of the k copies
    assert np.array_equal(S, np.repeat(x, k, axis=0))


def test_combine_single_choice_unit_weight_is_a_gather():
    rng = np.random.default_rng(7)
    Y = rng.integers(0, 0x7F00, size=(40, 16), dtype=np.uint16)
    dst = rng.permutation(40)[:25].astype(np.int32).reshape(25, 1)
    S, C = oracle.combine(Y, dst, np.ones((25, 1), np.float32))
    assert np.array_equal(S, Y[dst[:, 0]])
    assert np.array_equal(C, Y[dst[:, 0]])


def test_combine_hand_worked_exact_sums():
    # rows hold small integers, weights are powers of two: every product and
    # sum is exact, so C = sum_j w_j * Y[dst_j] can be written out by hand
    Y = _bf16_bits_from_f32(np.array([[1, 2, 3, 4], [8, 8, 8, 8], [-2, 0, 2, 6]], np.float32))
    dst = np.array([[1, 0], [2, 2]], np.int32)
    w = np.array([[0.5, 0.25], [1.0, 0.125]], np.float32)
    S, C = oracle.combine(Y, dst, w)
    want = np.array([[4.25, 4.5, 4.75, 5.0], [-2.25, 0.0, 2.25, 6.75]], np.float32)
    assert np.array_equal(C, _bf16_bits_from_f32(want))
    assert np.array_equal(S, Y[[1, 0, 2, 2]])


def test_combine_rounds_each_product_then_each_sum():
    # j=0 adds -(1 + 2^-7); j=1 multiplies (1 + 2^-23) by (1 + 2^-7) = 1 + 2^-7
    # + 2^-23 + 2^-30, which fp32 rounds to 1 + 2^-7 + 2^-23 before the add:
    # the sum is 2^-23.  A fused multiply-add would keep 2^-30 and give
    # 2^-23 * (1 + 2^-7), which bf16 represents, so the two readings differ.
    a = np.float32(1 + 2.0 ** -7)
    Y = _bf16_bits_from_f32(np.array([[-a], [a]], np.float32))
    w = np.array([[1.0, 1 + 2.0 ** -23]], np.float32)
    assert w[0, 1] != 1.0
    _, C = oracle.combine(Y, np.array([[0, 1]], np.int32), w)
    assert _f64_from_bits(C)[0, 0] == 2.0 ** -23


def test_combine_within_fp32_bound_of_float64():
    rng = np.random.default_rng(11)
    T, k, N, rows = 64, 4, 48, 300
    Y = _bf16_bits_from_f32(rng.standard_normal((rows, N)).astype(np.float32))
    dst = rng.integers(0, rows, size=(T, k)).astype(np.int32)
    logits = rng.standard_normal((T, k))
    w = (np.exp(logits) / np.exp(logits).sum(1, keepdims=True)).astype(np.float32)
    _, C = oracle.combine(Y, dst, w)
    Yf = _f64_from_bits(Y)
    exact = np.einsum("tj,tjn->tn", w.astype(np.float64), Yf[dst])
    mag = np.einsum("tj,tjn->tn", np.abs(w.astype(np.float64)), np.abs(Yf[dst]))
    got = _f64_from_bits(C)
    bound = 2 * k * 2.0 ** -24 * mag + 2.0 ** -8 * np.abs(exact) + 1e-30
    assert np.all(np.abs(got - exact) <= bound)


# ------------------------------------------------------------------ reduce-scatter
def test_reduce_partials_hand_worked():
    P = _bf16_bits_from_f32(np.array([[[1, 2, -3]], [[0.5, 2, 3]], [[0.25, -8, 1]]], np.float32))
    O = oracle.reduce_partials(P)
    assert np.array_equal(O, _bf16_bits_from_f32(np.array([[1.75, -4, 1]], np.float32)))


def test_reduce_partials_single_shard_is_identity():
    P = np.random.default_rng(3).integers(0, 0x7F00, size=(1, 17, 9), dtype=np.uint16)
    assert np.array_equal(oracle.reduce_partials(P), P[0])


def test_reduce_partials_accumulate_in_fp32():
    # 1 + 2^-8 + 2^-25 exactly lies just above the bf16 tie 1 + 2^-8 and rounds
    # up to 1 + 2^-7; in fp32 the 2^-25 (a quarter unit in the last place) is
    # lost in every order, the sum is the tie itself and rounds to even, 1.0
    P = _bf16_bits_from_f32(np.array([[[1.0]], [[2.0 ** -8]], [[2.0 ** -25]]], np.float32))
    assert _f64_from_bits(oracle.reduce_partials(P))[0, 0] == 1.0


def test_gemm_reduce_scatter_is_the_k_split_gemm():
    # small integers: every partial product is exact in bf16 and every sum in
    # fp32, so the shard sum equals the one GEMM over the whole K exactly
    rng = np.random.default_rng(4)
    S, M, Ks, N = 3, 10, 8, 12
    Xf = rng.integers(-2, 3, size=(S, M, Ks)).astype(np.float32)
    Wf = rng.integers(-2, 3, size=(S, Ks, N)).astype(np.float32)
    P, O = oracle.gemm_reduce_scatter(_bf16_bits_from_f32(Xf), _bf16_bits_from_f32(Wf))
    full = np.concatenate(list(Xf), axis=1) @ np.concatenate(list(Wf), axis=0)
    assert np.array_equal(_f64_from_bits(O), full)
    for s in range(S):
        assert np.array_equal(_f64_from_bits(P[s]), Xf[s] @ Wf[s])


def test_gemm_reduce_scatter_within_bound_of_float64():
    rng = np.random.default_rng(5)
    S, M, Ks, N = 4, 16, 64, 24
    X = _bf16_bits_from_f32(rng.standard_normal((S, M, Ks)).astype(np.float32))
    W = _bf16_bits_from_f32((rng.standard_normal((S, Ks, N)) / 8).astype(np.float32))
    _, O = oracle.gemm_reduce_scatter(X, W)
    Xd, Wd = _f64_from_bits(X), _f64_from_bits(W)
    exact = sum(Xd[s] @ Wd[s] for s in range(S))
    mag = sum(np.abs(Xd[s]) @ np.abs(Wd[s]) for s in range(S))
    # each partial: fp32 sum then bf16 rounding; then an fp32 sum of S terms and a final bf16 rounding
    bound = (Ks * 2.0 ** -24 + 2.0 ** -8) * mag + S * 2.0 ** -24 * mag + 2.0 ** -8 * np.abs(exact) + 1e-30
    assert np.all(np.abs(_f64_from_bits(O) - exact) <= bound)
