"""Static audit of CTA barriers in the CUDA sources (no GPU).

The sync-protocol page (section 6, item 4) warns that __syncthreads() is
hardware barrier 0 counting the whole CTA; if role-specialised warps use the
same id with another thread count, the result is undefined.  The kernels here
use barrier 0 (or, for CTA pairs, the cluster barrier) only at full-CTA
points -- before the role split and at teardown -- and warp roles coordinate
through mbarriers and a shared-memory hand-off.  The one other id: with
embedded copy warps, which skip the consumer prologue, the other warps meet
on barrier 1 with their own count (warps 0 .. 10); barrier 0 keeps the whole
CTA's count at every site.  This test pins that map."""
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "consumer_movement_gemm_gb300", "csrc")

# functions that run after the role split: no CTA-wide barrier may appear
ROLE_FUNCTIONS = {
    "consumer.cuh": ["consumer_tma", "consumer_mma", "consumer_epilogue", "gate", "consumer_gate", "wait_gate", "embedded_producer"],
    "producer.cuh": ["seed_counters", "begin_item", "load_pass", "store_pass", "copy_items", "copy_items_staged", "rs_reduce",
                     "rs_reduce_owned"],
    "copyplane.cuh": ["bulk_stream", "run_bulk"],
    "copy.cu": ["copy_v4", "copy_waiter", "copy_seeds"],
}
# full-CTA barrier sites allowed per function: (file, function) -> count
ALLOWED_SYNCTHREADS = {("consumer.cuh", "consumer"): 2, ("producer.cuh", "producer"): 1}
# (the consumer's third cluster barrier is the embedded copy warps' teardown)
ALLOWED_CLUSTER_SYNC = {("consumer.cuh", "consumer"): 3}
# explicit barrier ids: (file, function) -> the (id, thread count) arguments, in order
ALLOWED_BAR_SYNC = {("consumer.cuh", "consumer"): [("0", "kThreads"), ("1", "kFirstCopyWarp * 32"), ("0", "kThreads")]}


def _function_body(src: str, name: str) -> str:
    m = re.search(r"\b" + name + r"\s*\([^;{]*\)\s*\{", src)
    assert m, name
    i = m.end()
    depth = 1
    while depth:
        depth += {"{": 1, "}": -1}.get(src[i], 0)
        i += 1
    return src[m.end():i]


def test_named_barriers_only_at_audited_sites():
    for f in os.listdir(CSRC):
        text = open(os.path.join(CSRC, f)).read()
        assert not re.search(r"\bbar\.(sync|arrive|red)\b", text), f
        assert not re.search(r"\bbarrier\.(arrive|red)\b", text), f
        # the one barrier.sync instruction is the helper's
        if re.search(r"\bbarrier\.sync\b", text):
            assert f == "ptx.cuh", f
            assert len(re.findall(r"\bbarrier\.sync\b", text)) == 1
        calls = re.findall(r"bar_sync_unaligned\(([^,()]+),\s*([^;]+?)\);", text)
        if f == "ptx.cuh":
            continue
        want = [a for (ff, _), args in ALLOWED_BAR_SYNC.items() if ff == f for a in args]
        assert [(a.strip(), b.strip()) for a, b in calls] == want, f
    body = _function_body(open(os.path.join(CSRC, "consumer.cuh")).read(), "consumer")
    got = [(a.strip(), b.strip()) for a, b in re.findall(r"bar_sync_unaligned\(([^,()]+),\s*([^;]+?)\);", body)]
    assert got == ALLOWED_BAR_SYNC[("consumer.cuh", "consumer")]
    # barrier 1's count is the warps before the copy warps, which never reach it
    text = open(os.path.join(CSRC, "consumer.cuh")).read()
    assert "constexpr int kFirstCopyWarp = kGateWarp + 1;" in text
    assert "if (EMB && warp >= kFirstCopyWarp) {" in body


def test_no_cta_barrier_inside_roles():
    for f, names in ROLE_FUNCTIONS.items():
        text = open(os.path.join(CSRC, f)).read()
        for n in names:
            body = _function_body(text, n)
            assert "__syncthreads" not in body, (f, n)
            assert "cluster_sync" not in body, (f, n)


def test_cta_barrier_sites_are_the_audited_ones():
    for (f, n), count in ALLOWED_SYNCTHREADS.items():
        body = _function_body(open(os.path.join(CSRC, f)).read(), n)
        assert body.count("__syncthreads()") == count, (f, n)
    for (f, n), count in ALLOWED_CLUSTER_SYNC.items():
        body = _function_body(open(os.path.join(CSRC, f)).read(), n)
        assert body.count("cluster_sync()") == count, (f, n)
    # every CTA barrier after the role split is preceded by a warp reconvergence
    body = _function_body(open(os.path.join(CSRC, "consumer.cuh")).read(), "consumer")
    tail = body[body.index("consumer_tma<"):]
    assert tail.index("__syncwarp()") < tail.index("__syncthreads()")
    # the only cluster barrier instructions live in the one helper
    for f in os.listdir(CSRC):
        text = open(os.path.join(CSRC, f)).read()
        if "barrier.cluster" in text:
            assert f == "ptx.cuh", f
