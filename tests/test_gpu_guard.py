"""Guard bands around every buffer the path writes: each output (and the
workspace) sits inside a larger allocation whose 4 KiB bands before and after
it hold an all-ones byte pattern (NaN in bf16 and fp32).  After the pack,
attention forward, unpack and backward (two-kernel, or storing dS in the
workspace), the bands must be untouched: no kernel writes outside the rows,
heads or tiles it owns (ragged tails, replicated kv-heads, the ring hybrid and
D = 64 included)."""
import pytest
import torch

from pathcheck import GpuRun
from test_gpu_forward import wl
from ulysses_sequence_attention_seq_gb300 import binding as U

pytestmark = pytest.mark.gpu

BAND = 4096


class Guarded:
    def __init__(self, like: torch.Tensor):
        n = like.numel() * like.element_size()
        self.n = n
        self.raw = torch.full((n + 2 * BAND,), 0xFF, dtype=torch.uint8, device=like.device)
        self.t = self.raw[BAND:BAND + n].view(like.dtype).view(like.shape)

    def intact(self) -> bool:
        return bool((self.raw[:BAND] == 0xFF).all() and (self.raw[BAND + self.n:] == 0xFF).all())


CASES = [wl(2, 1, 424, 4, 2, 128),                              # ragged tail, GQA
         wl(4, 2, 512, 8, 8, 64, causal=False),                 # D = 64, B = 2
         wl(8, 1, 1024, 8, 2, 128),                             # kv-heads replicated (R = 4)
         wl(8, 1, 1024, 4, 4, 128).with_(ring=4),               # the ring hybrid, P > n_head
         wl(3, 1, 384, 2, 2, 64).with_(ring=3)]                 # hybrid, last tile pair past the end


@pytest.mark.parametrize("mode", ["two_kernel", "ds_store"])
@pytest.mark.parametrize("w", CASES, ids=lambda w: f"P{w.P}R{w.ring}B{w.B}S{w.S}h{w.n_head}kv{w.n_kv_head}D{w.head_dim}")
def test_no_write_outside_any_output(w, mode):
    w = w.with_(backward=True)
    ds = mode == "ds_store"
    run = GpuRun(w, backward=True, ds=ds)
    b, p = run.buf, run.prob
    g = {n: Guarded(getattr(b, n)) for n in ("q_head", "k_head", "v_head", "o_head", "lse", "o_seq",
                                             "dq_seq", "dk_seq", "dv_seq", "ws")}
    ws = g["ws"].t
    ws.copy_(b.ws)
    U.ulysses_pack_qkv(p, b.q_seq, b.k_seq, b.v_seq, g["q_head"].t, g["k_head"].t, g["v_head"].t, ws)
    U.ulysses_attn_fwd(p, g["q_head"].t, g["k_head"].t, g["v_head"].t, g["o_head"].t, g["lse"].t, ws)
    U.ulysses_unpack_out(p, g["o_head"].t, g["o_seq"].t)
    bwd = U.ulysses_attn_bwd_ds if ds else U.ulysses_attn_bwd
    bwd(p, g["q_head"].t, g["k_head"].t, g["v_head"].t, g["o_head"].t, g["lse"].t, b.do_seq,
        g["dq_seq"].t, g["dk_seq"].t, g["dv_seq"].t, ws)
    torch.cuda.synchronize()
    assert U.ulysses_read_status(ws) == 0
    bad = [n for n, x in g.items() if not x.intact()]
    assert not bad, f"writes outside: {bad}"
    # and the results are the ordinary path's
    run.forward()
    run.backward_ds() if ds else run.backward()
    for n in ("o_seq", "dq_seq", "dk_seq", "dv_seq"):
        assert torch.equal(g[n].t, getattr(b, n)), n
