"""GPU parity of the Ulysses x ring hybrid (the problem's `ring` field) against
the fp64 ring oracle (oracle/ring.py), through the C ABI.

The hybrid changes only who holds what: the All-to-All runs inside each ring
position, and the attention kernels read every ring position's key/value
chunk where the ring would circulate it.  So besides matching the oracle, each
output must be bit-identical to plain Ulysses over the same Pu-rank head split
(same tiles, same arithmetic, other addresses)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import ring as RG
from pathcheck import GpuRun, assert_close, assert_lse_close, oracle_inputs, oracle_problem, to64, ulp_bf16
from test_gpu_forward import sample_rows, wl
from ulysses_sequence_attention_seq_gb300 import binding as U
from ulysses_sequence_attention_seq_gb300.synthetic import EXTRA_WORKLOADS

pytestmark = pytest.mark.gpu


def rw(P, R, B, S, h, kv, D, causal=True, rope=True):
    return wl(P, B, S, h, kv, D, causal=causal, rope=rope).with_(ring=R)


RING_CASES = [rw(4, 2, 1, 512, 4, 2, 128),                  # 2 ring positions of 2 ranks
              rw(8, 4, 1, 1024, 4, 4, 64),                  # P = 8 > 4 heads
              rw(8, 8, 2, 1024, 2, 2, 128, causal=False),   # pure ring (one rank per position)
              rw(6, 3, 1, 768, 4, 2, 128),                  # three ring positions
              rw(3, 3, 1, 384, 2, 2, 64),                   # last query tile pair half past the end
              rw(8, 2, 1, 1024, 8, 2, 128),                 # kv-heads replicated inside a ring position
              rw(16, 4, 2, 1024, 4, 1, 64, causal=False)]   # one kv-head for the 4 members of every position


def _id(w):
    return f"P{w.P}R{w.ring}B{w.B}S{w.S}h{w.n_head}kv{w.n_kv_head}D{w.head_dim}{'c' if w.causal else 'n'}"


def _pack(run):
    b = run.buf
    U.ulysses_pack_qkv(run.prob, b.q_seq, b.k_seq, b.v_seq, b.q_head, b.k_head, b.v_head, b.ws)
    torch.cuda.synchronize()
    assert U.ulysses_read_status(b.ws) == 0


@pytest.mark.parametrize("w", RING_CASES, ids=_id)
def test_pack_is_the_ring_positions_all_to_all(w):
    """RoPE off: bit for bit the oracle's All-to-All inside each ring position;
    RoPE on: within one bf16 ulp of the fp64 rotation."""
    for rope in (False, True):
        wr = w.with_(use_rope=rope)
        run = GpuRun(wr)
        _pack(run)
        x = oracle_inputs(run.inputs)
        half = w.head_dim // 2
        for name, heads, got, rot in (("q", w.n_head, run.buf.q_head, rope), ("k", w.n_kv_head, run.buf.k_head, rope),
                                      ("v", w.n_kv_head, run.buf.v_head, False)):
            seq = oracle.shard_sequence(x[name], w.P)
            a2a = RG.a2a_seq_to_head_replicated if heads < w.P // w.ring else RG.a2a_seq_to_head
            want, _, _ = a2a(oracle.rope_seq(seq, float(np.float32(w.rope_base))) if rot else seq, heads, w.ring)
            # |x_i| + |x_{i+D/2}|: the size of what the fp32 rotation sums
            mag, _, _ = a2a([np.concatenate([np.abs(a[..., :half]) + np.abs(a[..., half:])] * 2, axis=-1)
                             for a in seq], heads, w.ring)
            g = to64(got)
            for r in range(w.P):
                if not rot:
                    assert np.array_equal(g[r], want[r]), f"{name} rank {r}"
                else:
                    assert np.all(np.abs(g[r] - want[r]) <= ulp_bf16(want[r]) + 2.0 ** -20 * mag[r]), \
                        f"{name} rank {r}"


@pytest.mark.parametrize("w", RING_CASES, ids=_id)
def test_unpack_is_bit_exact(w):
    prob = U.Problem.from_workload(w)
    g = torch.Generator().manual_seed(5)
    o_head_cpu = torch.randn(w.P, w.B, prob.Cs, prob.hp, w.head_dim, generator=g).to(prob.torch_dtype)
    o_seq = torch.empty(w.P, w.B, w.Sl, w.n_head * w.head_dim, dtype=prob.torch_dtype, device="cuda")
    U.ulysses_unpack_out(prob, o_head_cpu.cuda(), o_seq)
    torch.cuda.synchronize()
    want, _, _ = RG.a2a_head_to_seq([to64(o_head_cpu[r]) for r in range(w.P)], w.n_head, w.ring)
    got = to64(o_seq)
    for r in range(w.P):
        assert np.array_equal(got[r], want[r].reshape(w.B, w.Sl, -1))


@pytest.mark.parametrize("w", RING_CASES, ids=_id)
def test_forward_matches_ring_oracle(w):
    run = GpuRun(w)
    run.forward()
    x = oracle_inputs(run.inputs)
    want = RG.forward(oracle_problem(w), x["q"], x["k"], x["v"])
    got_o = to64(run.buf.o_seq)
    assert_close(got_o, np.stack([a.reshape(w.B, w.Sl, -1) for a in want["o_seq"]]), w, "o_seq")
    assert_lse_close(to64(run.buf.lse), np.stack(want["lse"]), w)


@pytest.mark.parametrize("w", RING_CASES, ids=_id)
def test_backward_matches_ring_oracle(w):
    """The two-kernel and the dS-store backward against the ring oracle; the
    dS-store one's dK and dV bit-identical to the two-kernel one's (the same
    kernel, which only also stores dS)."""
    w = w.with_(backward=True)
    run = GpuRun(w, backward=True, ds=True)
    run.forward()
    run.backward()
    x = oracle_inputs(run.inputs)
    want = RG.backward(oracle_problem(w), x["q"], x["k"], x["v"], x["do"])
    for name in ("dq_seq", "dk_seq", "dv_seq"):
        assert_close(to64(getattr(run.buf, name)), np.stack(want[name]), w, name)
    ref = {n: getattr(run.buf, n).clone() for n in ("dk_seq", "dv_seq")}
    for n in ("dq_seq", "dk_seq", "dv_seq"):
        getattr(run.buf, n).fill_(float("nan"))
    run.backward_ds()
    assert_close(to64(run.buf.dq_seq), np.stack(want["dq_seq"]), w, "dS-store dq_seq")
    for n, t in ref.items():
        assert torch.equal(getattr(run.buf, n), t), f"dS-store {n} differs from the two-kernel backward"


def _same_as_plain_ulysses(w, backward, ds=False):
    """The hybrid and plain Ulysses over Pu ranks compute every head with the
    same tiles in the same order: outputs equal bit for bit (sequence layout).
    With `ds`, the dS-store backward is compared too."""
    hyb = GpuRun(w, backward=backward, ds=ds)
    plain = GpuRun(w.with_(P=w.P // w.ring, ring=1), backward=backward, inputs=hyb.inputs, ds=ds)
    names = ("o_seq",) + (("dq_seq", "dk_seq", "dv_seq") if backward else ())

    def same(what):
        for name in names:
            a, b = getattr(hyb.buf, name), getattr(plain.buf, name)
            # both are [P][B][Sl][...] of the same global sequence, sharded P or P/ring ways
            assert torch.equal(a.reshape(-1), b.reshape(-1)) if w.B == 1 else \
                torch.equal(a.transpose(0, 1).reshape(w.B, -1), b.transpose(0, 1).reshape(w.B, -1)), (what, name)

    for run in (hyb, plain):
        run.forward()
        if backward:
            run.backward()
    same("two-kernel backward")
    if backward and ds:
        for run in (hyb, plain):
            for n in ("dq_seq", "dk_seq", "dv_seq"):
                getattr(run.buf, n).fill_(float("nan"))
            run.backward_ds()
        same("dS-store backward")


@pytest.mark.parametrize("w", RING_CASES[:3] + RING_CASES[5:], ids=_id)
def test_bit_identical_to_plain_ulysses(w):
    _same_as_plain_ulysses(w.with_(backward=True), backward=True, ds=True)


def test_full_size_pages_example():
    """The pages' head-count example at full size, in the bench's launch
    configuration: C4's model (32 heads, S = 32768) over P = 256 ranks as 8
    ring positions of 32.  Forward sampled against the ring oracle (every
    query row exact over its full key range), then forward and both the
    two-kernel and the dS-store backward bit-identical to plain Ulysses over
    32 ranks."""
    w = EXTRA_WORKLOADS["C4-ring8"]
    run = GpuRun(w, backward=False)
    run.forward()
    x = oracle_inputs(run.inputs)
    rows = sample_rows(w.with_(P=w.P // w.ring), 16, seed=3)
    rows = sorted(set(rows) | {c * (w.S // w.ring) + d for c in range(w.ring) for d in (-1, 0) if 0 <= c * (w.S // w.ring) + d})
    want = RG.forward(oracle_problem(w), x["q"], x["k"], x["v"], rows=rows)
    prob = run.prob
    got_h, got_lse = to64(run.buf.o_head), to64(run.buf.lse)
    for r in range(w.ring):
        mine = [p - r * prob.Cs for p in rows if r * prob.Cs <= p < (r + 1) * prob.Cs]
        for u in (0, prob.Pu // 2, prob.Pu - 1):
            me = r * prob.Pu + u
            assert_close(got_h[me][:, mine], want["o_head"][me][:, mine], w, f"o_head rank {me}")
            assert_lse_close(got_lse[me][..., mine], want["lse"][me][..., mine], w, f"lse rank {me}")
    del run, x, want
    torch.cuda.empty_cache()
    _same_as_plain_ulysses(w, backward=True, ds=True)
