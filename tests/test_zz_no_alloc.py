"""The routing plan entry point that allocates nothing.

tovl_dispatch_plan_noalloc is for callers that must not allocate device
memory (another framework owns the memory budget, a latency-critical loop
cannot afford cudaMalloc's device-wide synchronisation, a plugin's host owns
every allocation).  Its scratch is a fixed array inside the library, shared
by all calls on a device and keeping the previous call's contents.  This
file is collected last; it checks the entry point, through the C ABI, on two
calls in a row against the oracle's plan and against the plan the regular
dispatch entry point computes, and checks that a routing with a bad expert
id leaves all-zero offsets without spoiling the next call.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from consumer_movement_gemm_gb300 import tovl

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _build():
    from consumer_movement_gemm_gb300 import build
    build.build()
    oracle.build()


def _handle_plan(topk_np, E):
    """Expert offsets and destination rows from tovl_dispatch_grouped_gemm."""
    T, k = topk_np.shape
    H, N = 64, 256
    x = workloads.bf16_normal((T, H), 1 / math.sqrt(H), 1, DEV)
    W = workloads.bf16_normal((E, H, N), 1 / math.sqrt(H), 2, DEV)
    rows = tovl.dispatch_rows(T, k, E)
    with tovl.Handle(0, max_rows=rows, max_pairs=T * k, max_experts=E) as h:
        dispatched = torch.zeros(rows, H, dtype=torch.bfloat16, device=DEV)
        offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
        out = torch.empty(rows, N, dtype=torch.bfloat16, device=DEV)
        h.dispatch_grouped_gemm(x, torch.from_numpy(topk_np).to(DEV), W, dispatched, offs, out)
        assert h.sync_status() == 0
        _, dst, _, _, _, _ = h.read_plan(T, k, E)
    return offs.cpu().numpy(), dst


def _noalloc(topk_np, E):
    topk = torch.from_numpy(topk_np).to(DEV)
    offs = torch.full((E + 1,), -7, dtype=torch.int32, device=DEV)
    dst = torch.full((topk_np.size,), -7, dtype=torch.int32, device=DEV)
    tovl.dispatch_plan_noalloc(topk, E, offs, dst)
    torch.cuda.synchronize()
    return offs.cpu().numpy(), dst.cpu().numpy()


@pytest.mark.parametrize("routing", ["uniform", "zipf"])
def test_noalloc_plan_matches_oracle_and_dispatch_plan_twice(routing):
    if routing == "uniform":
        topk_np, E = workloads.uniform_topk(3000, 2, 8, 11), 8
    else:
        topk_np, E = workloads.zipf_topk(8192, 4, 32, 1.2, 12), 32
    want = oracle.dispatch_plan(topk_np, E)
    h_off, h_dst = _handle_plan(topk_np, E)
    for call in range(2):
        offs, dst = _noalloc(topk_np, E)
        # integer results: the tolerance is exact equality
        assert np.array_equal(offs, want.off), f"offsets vs oracle, call {call}"
        assert np.array_equal(dst, want.dst), f"destination rows vs oracle, call {call}"
        assert np.array_equal(offs, h_off), f"offsets vs the dispatch entry point, call {call}"
        assert np.array_equal(dst, h_dst), f"destination rows vs the dispatch entry point, call {call}"


def test_noalloc_bad_expert_id_gives_zero_offsets_and_next_call_is_clean():
    # an expert id outside [0, E) makes the plan all-zero offsets; the flag
    # that records it lives in the shared scratch, so the following valid
    # call must be cleared of it and agree with the oracle again
    E = 6
    bad = workloads.uniform_topk(500, 2, E, 13)
    bad[123, 1] = E
    offs, _ = _noalloc(bad, E)
    assert np.array_equal(offs, np.zeros(E + 1, np.int32))
    good = workloads.uniform_topk(700, 3, E, 14)
    want = oracle.dispatch_plan(good, E)
    offs, dst = _noalloc(good, E)
    assert np.array_equal(offs, want.off)
    assert np.array_equal(dst, want.dst)


def test_noalloc_plan_rejects_sizes_beyond_its_scratch():
    L = tovl.load()
    topk = torch.zeros(tovl_max_pairs() + 1, 1, dtype=torch.int32, device=DEV)
    offs = torch.empty(2, dtype=torch.int32, device=DEV)
    dst = torch.empty(topk.numel(), dtype=torch.int32, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    rc = L.tovl_dispatch_plan_noalloc(topk.data_ptr(), topk.shape[0], 1, 1, offs.data_ptr(), dst.data_ptr(), stream)
    assert rc == tovl.TOVL_ERR_UNSUPPORTED
    small = torch.zeros(4, 1, dtype=torch.int32, device=DEV)
    rc = L.tovl_dispatch_plan_noalloc(small.data_ptr(), 4, 1, 65, offs.data_ptr(), dst.data_ptr(), stream)
    assert rc == tovl.TOVL_ERR_UNSUPPORTED


def tovl_max_pairs() -> int:
    import os
    import re
    hdr = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "tovl.h")
    return int(re.search(r"#define TOVL_NOALLOC_MAX_PAIRS (\d+)", open(hdr).read()).group(1))
