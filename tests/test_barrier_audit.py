"""Static audit of CTA barriers in the CUDA sources (no GPU).

The sync-protocol page (section 6, item 4) warns that __syncthreads() is
hardware barrier 0 counting the whole CTA; if role-specialised warps use the
same id with another thread count, the result is undefined.  The kernels here
use barrier 0 (or, for CTA pairs, the cluster barrier) only at full-CTA
points -- before the role split and at teardown -- and warp roles coordinate
through mbarriers and a shared-memory hand-off.  The other ids: with embedded
copy warps, which skip the consumer prologue, the other warps (0 .. 10 and
the stage waiter, 15) meet on barrier 1 with their own count; and barriers
2 .. 2 + stages - 1 carry the stage hand-off from the stage waiter warp
(arrive) to the MMA warp (sync), 64 threads each, one id per pipeline stage.
Barrier 0 keeps the whole CTA's count at every site.  This test pins that
map."""
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "consumer_movement_gemm_gb300", "csrc")

# functions that run after the role split: no CTA-wide barrier may appear
ROLE_FUNCTIONS = {
    "consumer.cuh": ["consumer_tma", "consumer_mma", "consumer_stage_waiter", "consumer_epilogue", "gate", "consumer_gate",
                     "wait_gate", "embedded_producer"],
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
ALLOWED_BAR_SYNC = {("consumer.cuh", "consumer"): [("0", "kThreads"), ("1", "(kFirstCopyWarp + 1) * 32"), ("0", "kThreads")]}
# stage hand-off: (function, helper) pairs and their one argument list
STAGE_BARRIERS = {"consumer_mma": "bar_sync_aligned", "consumer_stage_waiter": "bar_arrive_aligned"}
STAGE_ARGS = ("kStageBar0 + static_cast<int>(stage)", "kStageBarThreads")


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
        assert not re.search(r"\bbarrier\.red\b", text), f
        # the barrier.sync / barrier.arrive instructions are the helpers'
        # (unaligned sync; aligned sync and arrive)
        if re.search(r"\bbarrier\.(sync|arrive)\b", text):
            assert f == "ptx.cuh", f
            assert len(re.findall(r"\bbarrier\.sync\b", text)) == 2
            assert len(re.findall(r"\bbarrier\.arrive\b", text)) == 1
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
    assert "if (EMB && warp >= kFirstCopyWarp && warp < kWaitWarp) {" in body


def test_stage_handoff_barriers():
    """Barriers 2 .. 2 + stages - 1: the waiter warp arrives, the MMA warp
    syncs, 64 threads (two whole warps), and no id collides with 0 or 1 or
    runs past the 16 a CTA has."""
    ctrl = open(os.path.join(CSRC, "ctrl.cuh")).read()
    consts = {k: int(v) for k, v in re.findall(r"constexpr int (k\w+) = (\d+);", ctrl)}
    assert consts["kStageBar0"] == 2 and consts["kStageBarThreads"] == 64
    assert consts["kWaitWarp"] == 15 and consts["kWaitWarp"] * 32 < consts["kThreads"]
    most = max(consts["kStages"], consts["kPairStages"], consts["kEmbPairStages"], consts["kWideStages"])
    assert consts["kStageBar0"] + most <= 16
    for f in os.listdir(CSRC):
        if f == "ptx.cuh":
            continue
        text = open(os.path.join(CSRC, f)).read()
        for helper in ("bar_sync_aligned", "bar_arrive_aligned"):
            n = len(re.findall(r"\b" + helper + r"\(", text))
            want = sum(1 for fn, h in STAGE_BARRIERS.items() if h == helper) if f == "consumer.cuh" else 0
            assert n == want, (f, helper, n)
    text = open(os.path.join(CSRC, "consumer.cuh")).read()
    for fn, helper in STAGE_BARRIERS.items():
        body = _function_body(text, fn)
        args = re.findall(helper + r"\(([^,()]+(?:\([^()]*\)[^,()]*)?),\s*([^;]+?)\);", body)
        assert [(a.strip(), b.strip()) for a, b in args] == [STAGE_ARGS], (fn, args)


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
