"""The measurement's own arithmetic (CPU): the algorithmic bytes a decode step must move
and the FLOPs of a prefill step (the numerators of bench.py's throughputs and roofline),
counted here token by token; the packing of a step's inputs for the end-to-end timing;
and the pipelined end-to-end loop's order, checked for races."""
import importlib.util
import os

import torch

from paged_kv_cache_90_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _brute_decode_bytes(w, st):
    """Walk every sequence, KV head and attended position; every table entry of a block
    holding an attended position; queries in and outputs out; one length per sequence."""
    elt = w.key_cache.element_size()
    W = w.sliding_window
    kv = tables = 0
    for L in st.context_lens.tolist():
        first = L - W if (W > 0 and L > W) else 0
        blocks = set()
        for pos in range(first, L):
            kv += w.num_kv_heads * 2 * w.head_dim * elt
            blocks.add(pos // w.block_size)
        tables += 4 * len(blocks) + 4
    q = st.query.numel() * st.query.element_size()
    return kv + 2 * q + tables


def test_decode_bytes_count_every_attended_token():
    b = _bench()
    for window in (0, 7, 16, 40):
        w = wl.variable_length_decode("acct", 3, [1, 5, 16, 17, 33, 100], 8, 2, 64, 16, "bf16", window=window)
        st = w.steps[0]
        assert b.decode_bytes(w, st) == _brute_decode_bytes(w, st), window
    w = wl.continuous_batching(seed=9, block_size=8, kv_dtype="e4m3", num_seqs=12, num_steps=1, median=40)
    assert b.decode_bytes(w, w.steps[0]) == _brute_decode_bytes(w, w.steps[0])


def test_mha_workload_counts_every_kv_head():
    """The multi-head workload (one query head per KV head) counts K and V of all 32 KV
    heads for every attended token."""
    b = _bench()
    w = b.make_workload("mha_decode")
    assert (w.num_heads, w.num_kv_heads, w.num_seqs) == (32, 32, 64)
    st = w.steps[0]
    assert b.decode_bytes(w, st) == _brute_decode_bytes(w, st)


def test_step_bytes_add_the_write_and_the_copies():
    b = _bench()
    w = wl.shared_prefix_cow(num_groups=2, group_size=4, prefix_blocks=2, suffix_range=(16, 60))
    st = w.steps[0]
    elt = w.key_cache.element_size()
    t = st.slot_mapping.numel()
    write = 2 * st.new_key.numel() * st.new_key.element_size() + 8 * t + 2 * t * w.num_kv_heads * w.head_dim * elt
    pairs = st.cow_pairs.shape[0]
    assert pairs > 0
    block = w.num_kv_heads * w.block_size * w.head_dim * elt
    cow = pairs * (2 * 2 * block + 16)                  # read + write, K and V; the pair itself
    assert b.step_bytes(w, st) == b.decode_bytes(w, st) + write + cow


def test_prefill_flops_count_every_causal_pair():
    b = _bench()
    w = wl.chunked_prefill()
    st = w.steps[0]
    qsl = st.query_start_loc.tolist()
    pairs = 0
    for s, L in enumerate(st.context_lens.tolist()):
        n = qsl[s + 1] - qsl[s]
        for i in range(n):                              # new token i at position L - n + i
            pairs += L - n + i + 1
    assert b.prefill_flops(w, st) == 4 * w.head_dim * w.num_heads * pairs


def test_staged_inputs_round_trip(monkeypatch):
    """Every field packed into one buffer at a 256-byte aligned offset and viewed back
    with its dtype and shape (pinning is a no-op here: no GPU)."""
    b = _bench()
    monkeypatch.setattr(torch.Tensor, "pin_memory", lambda self: self)
    for w, fields in ((wl.shared_prefix_cow(num_groups=2, prefix_blocks=2), b.DeviceStep.__dataclass_fields__),
                      (wl.chunked_prefill(), b.DeviceStep.__dataclass_fields__)):
        st = w.steps[0]
        names = tuple(f for f in fields if getattr(st, f, None) is not None)
        host, dev, views, nbytes = b.staged_inputs(st, names, "cpu")
        dev.copy_(host)
        assert nbytes == sum(getattr(st, f).numel() * getattr(st, f).element_size() for f in names)
        for f in names:
            v = getattr(views, f)
            assert v.dtype == getattr(st, f).dtype and v.shape == getattr(st, f).shape
            assert torch.equal(v, getattr(st, f)), f
            if v.numel():
                assert (v.data_ptr() - dev.data_ptr()) % 256 == 0


def test_profile_digest_covers_existing_sources():
    b = _bench()
    csrc = os.path.join(ROOT, "paged_kv_cache_90_gb300", "csrc")
    for name in b.DECODE_SOURCES:
        assert os.path.exists(os.path.join(csrc, name)), name
    assert len(b.source_digest()) == 16


def _happens_before(ops):
    """For each op of a two-stream schedule, the set of ops certain to finish before it
    starts: a stream runs its ops in issue order, and a wait on an event follows the
    last op its stream issued before the event was recorded (a wait must come after its
    record in issue order, as for CUDA events)."""
    before, last, rec = [], {}, {}
    for i, (where, op, k) in enumerate(ops):
        preds = set()
        if where in last:
            preds.add(last[where])
        last[where] = i
        if op.startswith("record_"):
            rec[(op[len("record_"):], k)] = i
        if op.startswith("wait_"):
            preds.add(rec[(op[len("wait_"):], k)])
        s = set()
        for p in preds:
            s |= before[p]
            s.add(p)
        before.append(s)
    return before


def _pipeline_hazards(ops, nbuf):
    """Races of the pipelined end-to-end loop: a step's call not behind its input copy,
    an input copy overwriting a buffer an earlier call may still read, a call writing an
    output buffer whose earlier output copy may still run, an output copy not behind its
    call."""
    before = _happens_before(ops)
    at = {(op, k): i for i, (_, op, k) in enumerate(ops)}
    steps = sorted({k for _, op, k in ops if op == "call"})
    bad = []
    for k in steps:
        if at[("h2d", k)] not in before[at[("call", k)]]:
            bad.append(("call before its input", k))
        if at[("call", k)] not in before[at[("d2h", k)]]:
            bad.append(("output copied before its call", k))
        for m in steps:
            if m < k and m % nbuf == k % nbuf and at[("call", m)] not in before[at[("h2d", k)]]:
                bad.append(("input buffer overwritten while read", m, k))
            if m < k and m % 2 == k % 2 and at[("d2h", m)] not in before[at[("call", k)]]:
                bad.append(("output buffer written while copied", m, k))
    return bad


def test_e2e_pipeline_has_no_buffer_races():
    """The pipelined end-to-end schedule, checked for every race between its copies and
    its calls, with two or more (even) input buffers and two output buffers."""
    b = _bench()
    for count in (1, 2, 3, 4, 10, 25):
        ops = b.e2e_pipeline_ops(count)
        assert sorted(k for _, op, k in ops if op == "call") == list(range(count))
        assert sum(op == "h2d" for _, op, _ in ops) == count and sum(op == "d2h" for _, op, _ in ops) == count
        for nbuf in (2, 4, 10, 20):
            assert _pipeline_hazards(ops, nbuf) == [], (count, nbuf)


def test_e2e_race_check_catches_broken_schedules():
    """The race check itself: one input buffer, output copies issued without waiting for
    their calls, and input copies issued two steps ahead are each caught."""
    b = _bench()
    ops = b.e2e_pipeline_ops(6)
    assert ("input buffer overwritten while read", 0, 1) in _pipeline_hazards(ops, 1)
    no_wait = [x for x in ops if x[1] != "wait_done"]
    assert ("output copied before its call", 0) in _pipeline_hazards(no_wait, 2)
    ahead = [("copy", "h2d", 0), ("copy", "record_in", 0), ("copy", "h2d", 1), ("copy", "record_in", 1)]
    for k in range(6):
        if k + 2 < 6:
            ahead += [("copy", "h2d", k + 2), ("copy", "record_in", k + 2)]
        ahead += [("compute", "wait_in", k), ("compute", "call", k), ("compute", "record_done", k),
                  ("copy", "wait_done", k), ("copy", "d2h", k)]
    hazards = _pipeline_hazards(ahead, 2)
    assert ("input buffer overwritten while read", 0, 2) in hazards
    assert ("output buffer written while copied", 0, 2) in hazards
