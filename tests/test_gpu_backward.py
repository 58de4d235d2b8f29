"""GPU parity of the backward path (dO seq->head + delta, tensor-core dK/dV and
dQ, reverse All-to-All with the RoPE rotation undone) against the fp64
oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from pathcheck import GpuRun, assert_close, oracle_inputs, oracle_problem, to64
from test_gpu_forward import sample_rows, wl
from ulysses_sequence_attention_seq_gb300 import binding as U
from ulysses_sequence_attention_seq_gb300.synthetic import WORKLOADS

pytestmark = pytest.mark.gpu

BWD_CASES = [wl(2, 1, 424, 4, 2, 128),                       # ragged tail, GQA 2
             wl(4, 2, 512, 8, 8, 64),                        # D = 64, B = 2
             wl(2, 1, 320, 2, 2, 128, causal=False, rope=False),
             wl(1, 1, 640, 4, 1, 128),                       # P = 1, 4 q-heads per kv-head
             wl(8, 1, 1024, 32, 8, 128),                     # the GQA workload's head layout
             wl(2, 1, 200, 4, 4, 64, causal=False)]


def _ids(w):
    return f"P{w.P}B{w.B}S{w.S}h{w.n_head}kv{w.n_kv_head}D{w.head_dim}{'c' if w.causal else 'n'}{'r' if w.use_rope else ''}"


@pytest.mark.parametrize("w", BWD_CASES, ids=_ids)
def test_backward_matches_oracle(w):
    w = w.with_(backward=True)
    run = GpuRun(w, backward=True)
    run.forward()
    run.backward()
    x = oracle_inputs(run.inputs)
    want = oracle.backward(oracle_problem(w), x["q"], x["k"], x["v"], x["do"])
    for name in ("dq_seq", "dk_seq", "dv_seq"):
        got = to64(getattr(run.buf, name))
        assert_close(got, np.stack(want[name]), w, name)


def test_backward_is_deterministic():
    w = wl(4, 1, 1024, 8, 4, 128).with_(backward=True)
    run = GpuRun(w, backward=True)
    run.forward()
    outs = []
    for _ in range(3):
        run.backward()
        outs.append([getattr(run.buf, n).clone() for n in ("dq_seq", "dk_seq", "dv_seq")])
    for o in outs[1:]:
        for a, b in zip(o, outs[0]):
            assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["C3", "C4"])
def test_backward_workloads(name):
    """Full-size backward, sampled: two (rank, kv-head) groups (the first and
    the last), every gradient row at shard/tile boundaries and seeded random
    rows, each exact over its full key or query range."""
    w = WORKLOADS[name]
    run = GpuRun(w, backward=True)
    run.forward()
    run.backward()
    x = oracle_inputs(run.inputs)
    rows = sample_rows(w, 16, seed=1)
    kvp = w.n_kv_head // w.P
    groups = [(0, 0, 0), (w.P - 1, w.B - 1, kvp - 1)]
    want = oracle.backward(oracle_problem(w), x["q"], x["k"], x["v"], x["do"], groups=groups,
                           q_rows=rows, kv_rows=rows)
    # compare in head layout: rank r, local heads of the sampled groups
    G = w.n_head // w.n_kv_head
    hp = w.n_head // w.P
    got_seq = {n: to64(getattr(run.buf, n)) for n in ("dq_seq", "dk_seq", "dv_seq")}
    for (r, b, kl) in groups:
        kv_glob = r * kvp + kl
        for name, heads in (("dk_seq", [kv_glob]), ("dv_seq", [kv_glob]),
                            ("dq_seq", [r * hp + kl * G + gi for gi in range(G)])):
            got = np.concatenate(list(got_seq[name]), axis=1)     # [B][S][heads][D] global
            ref = np.concatenate(list(want[name]), axis=1)
            sel_g = got[b][rows][:, heads]
            sel_r = ref[b][rows][:, heads]
            assert_close(sel_g, sel_r, w, f"{name} rank {r} kv-head {kl}")


@pytest.mark.parametrize("order", ["dkdv_first", "dq_first"])
def test_backward_steps_equal_composed_call(order):
    """ulysses_attn_bwd_prepare + _dkdv + _dq (either order of the last two)
    give exactly what ulysses_attn_bwd gives."""
    w = WORKLOADS["C3"].with_(S=1024)
    run = GpuRun(w, backward=True)
    run.forward()
    run.backward()
    b = run.buf
    ref = [t.clone() for t in (b.dq_seq, b.dk_seq, b.dv_seq)]
    for t in (b.dq_seq, b.dk_seq, b.dv_seq):
        t.zero_()
    U.ulysses_attn_bwd_prepare(run.prob, b.o_head, b.lse, b.do_seq, b.ws)
    steps = [lambda: U.ulysses_attn_bwd_dkdv(run.prob, b.q_head, b.k_head, b.v_head, b.dk_seq, b.dv_seq, b.ws),
             lambda: U.ulysses_attn_bwd_dq(run.prob, b.q_head, b.k_head, b.v_head, b.dq_seq, b.ws)]
    for f in (steps if order == "dkdv_first" else steps[::-1]):
        f()
    torch.cuda.synchronize()
    assert U.ulysses_read_status(b.ws) == 0
    for got, want in zip((b.dq_seq, b.dk_seq, b.dv_seq), ref):
        assert torch.equal(got, want)


# KV-head replication: each replica computes dK, dV for its own q-heads; the
# kv-head's gradient is their sum (deterministic, in rank order).
REP_BWD_CASES = [wl(4, 1, 512, 8, 2, 128),                  # R = 2
                 wl(8, 1, 1024, 8, 1, 64),                  # R = 8 (MQA)
                 wl(8, 2, 392, 16, 4, 128, causal=False)]   # R = 2, B = 2, ragged tail


@pytest.mark.parametrize("w", REP_BWD_CASES, ids=_ids)
def test_replicated_kv_backward_matches_oracle(w):
    w = w.with_(backward=True)
    run = GpuRun(w, backward=True)
    run.forward()
    run.backward()
    x = oracle_inputs(run.inputs)
    want = oracle.backward(oracle_problem(w), x["q"], x["k"], x["v"], x["do"])
    for name in ("dq_seq", "dk_seq", "dv_seq"):
        assert_close(to64(getattr(run.buf, name)), np.stack(want[name]), w, name)


def test_replicated_kv_backward_is_deterministic():
    w = wl(8, 1, 512, 8, 2, 128).with_(backward=True)
    run = GpuRun(w, backward=True)
    run.forward()
    outs = []
    for _ in range(2):
        run.backward()
        outs.append([getattr(run.buf, n).clone() for n in ("dq_seq", "dk_seq", "dv_seq")])
    for a, b in zip(outs[1], outs[0]):
        assert torch.equal(a, b)


def test_replicated_kv_backward_full_size_sampled():
    """The replicated workload at full size (the bench's launch configuration),
    sampled: kv-head 0 and the last kv-head with every replica rank of each
    (their partials are what the sum needs), gradient rows at shard/tile
    boundaries and seeded random rows, each exact over its full range."""
    from ulysses_sequence_attention_seq_gb300.synthetic import EXTRA_WORKLOADS
    w = EXTRA_WORKLOADS["C4-kv4"]
    run = GpuRun(w, backward=True)
    run.forward()
    run.backward()
    x = oracle_inputs(run.inputs)
    rows = sample_rows(w, 12, seed=2)
    R = w.P // w.n_kv_head
    kvs = [0, w.n_kv_head - 1]
    groups = [(kv * R + j, 0, 0) for kv in kvs for j in range(R)]
    want = oracle.backward(oracle_problem(w), x["q"], x["k"], x["v"], x["do"], groups=groups,
                           q_rows=rows, kv_rows=rows)
    hp = w.n_head // w.P
    for name, heads in (("dk_seq", kvs), ("dv_seq", kvs),
                        ("dq_seq", [r * hp + j for (r, _, _) in groups for j in range(hp)])):
        got = np.concatenate(list(to64(getattr(run.buf, name))), axis=1)   # [B][S][heads][D] global
        ref = np.concatenate(list(want[name]), axis=1)
        assert_close(got[0][rows][:, heads], ref[0][rows][:, heads], w, name)
