"""The routing plan entry point that allocates nothing.

tovl_dispatch_plan_noalloc is for callers that must not allocate device
memory (another framework owns the memory budget, a latency-critical loop
cannot afford cudaMalloc's device-wide synchronisation, a plugin's host owns
every allocation).  Its scratch is a fixed array inside the library, shared
by all calls on a device and keeping the previous call's contents.  This
file is collected last; it checks the entry point, through the C ABI, against
the plan the regular dispatch entry point computes, on two calls in a row.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from consumer_movement_gemm_gb300 import tovl

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _build():
    from consumer_movement_gemm_gb300 import build
    build.build()


def _reference_plan(topk_np, E):
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


@pytest.mark.parametrize("routing", ["uniform", "zipf"])
def test_noalloc_plan_matches_dispatch_plan_twice(routing):
    if routing == "uniform":
        topk_np, E = workloads.uniform_topk(3000, 2, 8, 11), 8
    else:
        topk_np, E = workloads.zipf_topk(8192, 4, 32, 1.2, 12), 32
    want_off, want_dst = _reference_plan(topk_np, E)
    topk = torch.from_numpy(topk_np).to(DEV)
    for call in range(2):
        offs = torch.full((E + 1,), -7, dtype=torch.int32, device=DEV)
        dst = torch.full((topk_np.size,), -7, dtype=torch.int32, device=DEV)
        tovl.dispatch_plan_noalloc(topk, E, offs, dst)
        torch.cuda.synchronize()
        # integer results: the tolerance is exact equality
        assert np.array_equal(offs.cpu().numpy(), want_off), f"offsets, call {call}"
        assert np.array_equal(dst.cpu().numpy(), want_dst), f"destination rows, call {call}"


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
