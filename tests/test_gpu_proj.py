"""GPU parity of the fused QKV projection + pack + RoPE (ulysses_qkv_proj_pack)
against the oracle's per-rank projection, RoPE and All-to-All, through the C
ABI.  Sizes span several 128 x 256 tiles with ragged token and feature tails."""
import numpy as np
import pytest
import torch

import oracle
from pathcheck import assert_close, oracle_problem, to64
from test_gpu_forward import sample_rows, wl
from ulysses_sequence_attention_seq_gb300 import binding as U

pytestmark = pytest.mark.gpu


def _weights(w, bias, seed):
    g = torch.Generator().manual_seed(seed)
    H, N = w.hidden, (w.n_head + 2 * w.n_kv_head) * w.head_dim
    x = torch.randn(w.B, w.S, H, generator=g).to(torch.bfloat16)
    W = (torch.randn(N, H, generator=g) / H ** 0.5).to(torch.bfloat16)
    b = (0.1 * torch.randn(N, generator=g)).to(torch.bfloat16) if bias else None
    return x, W, b


def _run(w, x, W, b):
    prob = U.Problem.from_workload(w)
    buf = U.Buffers(prob)
    dev = buf.q_head.device
    x_seq = U.seq_layout(x, w.P).to(dev)
    Wd = W.to(dev)
    bd = b.to(dev) if b is not None else None
    U.ulysses_workspace_init(prob, buf.ws)
    U.ulysses_qkv_proj_pack(prob, x_seq, Wd, bd, buf.q_head, buf.k_head, buf.v_head, buf.ws)
    torch.cuda.synchronize()
    assert U.ulysses_read_status(buf.ws) == 0
    return buf


CASES = [wl(2, 1, 424, 4, 2, 128),                         # ragged token tail, 4 feature tiles
         wl(4, 2, 256, 8, 8, 64, rope=False),              # D = 64, no RoPE
         wl(1, 1, 300, 3, 1, 128),                         # 5 heads of output: a half feature tile
         wl(4, 1, 512, 8, 2, 128),                         # replicated kv-heads (R = 2)
         wl(8, 1, 1024, 32, 8, 128, causal=False)]         # the GQA workload's head layout


@pytest.mark.parametrize("bias", [True, False])
@pytest.mark.parametrize("w", CASES, ids=lambda w: f"P{w.P}B{w.B}S{w.S}h{w.n_head}kv{w.n_kv_head}D{w.head_dim}{'r' if w.use_rope else ''}")
def test_qkv_proj_pack_matches_oracle(w, bias):
    x, W, b = _weights(w, bias, 5)
    buf = _run(w, x, W, b)
    prob = oracle_problem(w)
    xs = oracle.shard_sequence(to64(x), w.P)
    qh, kh, vh = oracle.project_and_pack(prob, xs, to64(W), None if b is None else to64(b))
    for name, got, want in (("q_head", buf.q_head, qh), ("k_head", buf.k_head, kh), ("v_head", buf.v_head, vh)):
        assert_close(to64(got), np.stack(want), w, name)


def test_qkv_proj_pack_full_size_sampled():
    """The pages' sizing (P=8, S=32768, hidden 4096, 32 heads, D=128, RoPE) in
    the launch configuration the bench times, on sampled tokens of every rank:
    each sampled output row is the exact fp64 projection of its token, rotated
    at its global position."""
    from ulysses_sequence_attention_seq_gb300.synthetic import WORKLOADS
    w = WORKLOADS["C4"]
    x, W, b = _weights(w, True, 9)
    buf = _run(w, x, W, b)
    rows = sample_rows(w, 64, seed=3)
    D, h, kv, hp = w.head_dim, w.n_head, w.n_kv_head, w.n_head // w.P
    x64, W64, b64 = to64(x), to64(W), to64(b)
    y = (x64[0, rows] @ W64.T + b64[None, :]).reshape(len(rows), h + 2 * kv, D)
    q = oracle.rope_rows(y[:, :h], rows, w.rope_base)
    k = oracle.rope_rows(y[:, h:h + kv], rows, w.rope_base)
    v = y[:, h + kv:]
    kvp = kv // w.P
    rows_t = torch.tensor(rows, device=buf.q_head.device)
    for hd in range(h):
        assert_close(to64(buf.q_head[hd // hp, 0, rows_t, hd % hp]), q[:, hd], w, f"q head {hd}")
    for hd in range(kv):
        assert_close(to64(buf.k_head[hd // kvp, 0, rows_t, hd % kvp]), k[:, hd], w, f"k head {hd}")
        assert_close(to64(buf.v_head[hd // kvp, 0, rows_t, hd % kvp]), v[:, hd], w, f"v head {hd}")


OUT_CASES = [wl(2, 1, 512, 4, 4, 128),                      # 4 x 2 tiles
             wl(4, 2, 1024, 8, 8, 64),                      # D = 64, B = 2
             wl(1, 1, 256, 3, 1, 128, rope=False),          # hidden 384: a half feature tile
             wl(8, 1, 2048, 32, 8, 128)]                    # the GQA workload's head layout


@pytest.mark.parametrize("bias", [True, False])
@pytest.mark.parametrize("w", OUT_CASES, ids=lambda w: f"P{w.P}B{w.B}S{w.S}h{w.n_head}D{w.head_dim}")
def test_out_proj_unpack_matches_oracle(w, bias):
    prob = U.Problem.from_workload(w)
    buf = U.Buffers(prob)
    dev = buf.q_head.device
    g = torch.Generator().manual_seed(13)
    H = w.hidden
    o_head = torch.randn(w.P, w.B, w.S, w.n_head // w.P, w.head_dim, generator=g).to(torch.bfloat16)
    W = (torch.randn(H, H, generator=g) / H ** 0.5).to(torch.bfloat16)
    b = (0.1 * torch.randn(H, generator=g)).to(torch.bfloat16) if bias else None
    y = torch.empty(w.P, w.B, w.Sl, H, dtype=torch.bfloat16, device=dev)
    U.ulysses_workspace_init(prob, buf.ws)
    U.ulysses_out_proj_unpack(prob, o_head.to(dev), W.to(dev), None if b is None else b.to(dev), y, buf.ws)
    torch.cuda.synchronize()
    assert U.ulysses_read_status(buf.ws) == 0
    want = oracle.unpack_and_project(oracle_problem(w), list(to64(o_head)), to64(W), None if b is None else to64(b))
    assert_close(to64(y), np.stack(want), w, "y_seq")


def test_out_proj_unpack_full_size_sampled():
    """The pages' sizing (P=8, S=32768, hidden 4096) in the launch
    configuration the bench times, on sampled tokens of every rank."""
    from ulysses_sequence_attention_seq_gb300.synthetic import WORKLOADS
    w = WORKLOADS["C4"]
    prob = U.Problem.from_workload(w)
    buf = U.Buffers(prob)
    dev = buf.q_head.device
    g = torch.Generator().manual_seed(17)
    H, hp, D = w.hidden, w.n_head // w.P, w.head_dim
    o_head = torch.randn(w.P, w.B, w.S, hp, D, generator=g).to(torch.bfloat16)
    W = (torch.randn(H, H, generator=g) / H ** 0.5).to(torch.bfloat16)
    b = (0.1 * torch.randn(H, generator=g)).to(torch.bfloat16)
    y = torch.empty(w.P, w.B, w.Sl, H, dtype=torch.bfloat16, device=dev)
    U.ulysses_workspace_init(prob, buf.ws)
    U.ulysses_out_proj_unpack(prob, o_head.to(dev), W.to(dev), b.to(dev), y, buf.ws)
    torch.cuda.synchronize()
    assert U.ulysses_read_status(buf.ws) == 0
    rows = sample_rows(w, 48, seed=4)
    o64 = to64(o_head)
    # token p's feature vector: head hd comes from rank hd // hp, local head hd % hp
    x = np.stack([np.concatenate([o64[hd // hp, 0, pos, hd % hp] for hd in range(w.n_head)]) for pos in rows])
    want = x @ to64(W).T + to64(b)[None, :]
    got = np.stack([to64(y[pos // w.Sl, 0, pos % w.Sl]) for pos in rows])
    assert_close(got, want, w, "y rows")


@pytest.mark.parametrize("w", [wl(2, 1, 512, 4, 2, 128), wl(4, 1, 1024, 8, 2, 64, causal=False)],
                         ids=lambda w: f"P{w.P}S{w.S}h{w.n_head}kv{w.n_kv_head}D{w.head_dim}")
def test_attention_layer_forward_matches_oracle(w):
    """The whole Ulysses attention layer through the C ABI -- QKV projection
    with the pack and RoPE, attention, output projection with the unpack --
    against the oracle's steps in the pages' order."""
    prob = U.Problem.from_workload(w)
    buf = U.Buffers(prob)
    dev = buf.q_head.device
    x, W, b = _weights(w, True, 21)
    g = torch.Generator().manual_seed(22)
    H = w.hidden
    Wo = (torch.randn(H, H, generator=g) / H ** 0.5).to(torch.bfloat16)
    bo = (0.1 * torch.randn(H, generator=g)).to(torch.bfloat16)
    y = torch.empty(w.P, w.B, w.Sl, H, dtype=torch.bfloat16, device=dev)
    U.ulysses_workspace_init(prob, buf.ws)
    U.ulysses_qkv_proj_pack(prob, U.seq_layout(x, w.P).to(dev), W.to(dev), b.to(dev), buf.q_head, buf.k_head,
                            buf.v_head, buf.ws)
    U.ulysses_attn_fwd(prob, buf.q_head, buf.k_head, buf.v_head, buf.o_head, buf.lse, buf.ws)
    U.ulysses_out_proj_unpack(prob, buf.o_head, Wo.to(dev), bo.to(dev), y, buf.ws)
    torch.cuda.synchronize()
    assert U.ulysses_read_status(buf.ws) == 0
    op = oracle_problem(w)
    qh, kh, vh = oracle.project_and_pack(op, oracle.shard_sequence(to64(x), w.P), to64(W), to64(b))
    o_head, _ = oracle.attention_fwd(op, qh, kh, vh)
    want = oracle.unpack_and_project(op, o_head, to64(Wo), to64(bo))
    assert_close(to64(y), np.stack(want), w, "layer y")
