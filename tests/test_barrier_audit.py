"""Static audit of CTA barriers in the CUDA sources (no GPU).

The sync-protocol page (section 6, item 4) warns that __syncthreads() is
hardware barrier 0 counting the whole CTA; if role-specialised warps use the
same id with another thread count, the result is undefined.  The kernels here
use barrier 0 only at full-CTA points -- before the role split and at
teardown -- and no named barriers at all; warp roles coordinate through
mbarriers.  This test pins that map."""
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "consumer_movement_gemm_gb300", "csrc")

# functions that run after the role split: no CTA-wide barrier may appear
ROLE_FUNCTIONS = {
    "fused.cu": ["consumer_tma", "consumer_mma", "consumer_epilogue", "gate", "seed_counters", "copy_item"],
    "copyplane.cuh": ["bulk_stream", "run_bulk"],
    "copy.cu": ["copy_v4", "copy_waiter", "copy_seeds"],
}
# full-CTA barrier-0 sites allowed per function
ALLOWED_SYNCTHREADS = {("fused.cu", "consumer"): 2, ("fused.cu", "producer"): 1}


def _function_body(src: str, name: str) -> str:
    m = re.search(r"\b" + name + r"\s*\([^;{]*\)\s*\{", src)
    assert m, name
    i = m.end()
    depth = 1
    while depth:
        depth += {"{": 1, "}": -1}.get(src[i], 0)
        i += 1
    return src[m.end():i]


def test_no_named_barriers():
    for f in os.listdir(CSRC):
        text = open(os.path.join(CSRC, f)).read()
        assert not re.search(r"\bbar(rier)?\.(sync|arrive|red)\b", text), f
        assert "named_barrier" not in text, f


def test_no_cta_barrier_inside_roles():
    for f, names in ROLE_FUNCTIONS.items():
        text = open(os.path.join(CSRC, f)).read()
        for n in names:
            assert "__syncthreads" not in _function_body(text, n), (f, n)


def test_cta_barrier_sites_are_the_audited_ones():
    text = open(os.path.join(CSRC, "fused.cu")).read()
    for (f, n), count in ALLOWED_SYNCTHREADS.items():
        body = _function_body(open(os.path.join(CSRC, f)).read(), n)
        assert body.count("__syncthreads()") == count, (f, n)
    # every CTA barrier in the consumer is preceded by a warp reconvergence or
    # sits before the role split
    body = _function_body(text, "consumer")
    split = body.index("consumer_tma(")
    tail = body[split:]
    assert tail.index("__syncwarp()") < tail.index("__syncthreads()")
