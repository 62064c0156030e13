"""The library's calls inside CUDA graphs: a step of cross-entropy, fused
linear + CE and fused linear + JSD calls (forward and backward, and the
vocab-parallel merges) is captured once into a torch.cuda.CUDAGraph and
replayed; every replay must give the eager calls' results bit for bit, also
after new inputs are copied into the captured buffers.

Everything the graph touches is allocated before the capture (outputs and
zero-filled workspaces passed explicitly), and each call runs once eagerly
first, so the one-time host set-up (shared-memory limits, the tensor-map
encoder, cluster occupancy) happens outside the capture.  The calls only
enqueue kernels on the current stream and leave their workspaces' zero words
at zero, which is what makes a replayed graph equal to a fresh call."""
import numpy as np
import pytest
import torch

import gen
from tests.helpers import to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


class Step:
    """Static inputs, outputs and workspaces of one captured step."""

    def __init__(self, lmho, seed):
        self.lmho = lmho
        T, V = 512, 4096
        self.z = to_dev(gen.normal_f32(seed, 0, (T, V)))
        self.t = to_dev(gen.targets(seed, 1, (T,), V))
        self.zb = to_dev_bf16(gen.normal_bf16_bits(seed, 0, (64, 4, 3000), sigma=2.0))
        self.tb = to_dev(gen.targets(seed, 1, (64, 4), 3000))
        Tf, H, Vf = 256, 256, 3000
        self.x = to_dev_bf16(gen.normal_bf16_bits(seed, 2, (Tf, H)))
        self.W = to_dev_bf16(gen.normal_bf16_bits(seed, 3, (Vf, H), sigma=0.1))
        self.xt = to_dev_bf16(gen.normal_bf16_bits(seed, 4, (Tf, H)))
        self.Wt = to_dev_bf16(gen.normal_bf16_bits(seed, 5, (Vf, H), sigma=0.1))
        self.tt = to_dev(gen.targets(seed, 6, (Tf,), Vf))
        self.keep = to_dev((np.arange(Tf) % 5 != 2).astype(np.uint8))
        f = lambda *shape: torch.full(shape, float("nan"), device="cuda")
        self.out = dict(ce=f(1), sbv=f(64, 4), flce=f(1), dx=f(Tf, H), dW=f(Vf, H), jsd=f(1), dxs=f(Tf, H),
                        dWs=f(Vf, H), parts=f(2, 3, Tf), vp_rows=f(Tf), vp_mean=f(1))
        self.ws = dict(ce=lmho.workspace(lmho.ce_workspace_bytes(T, V)),
                       flce=lmho.workspace(lmho.flce_bwd_workspace_bytes(Tf, H, Vf)),
                       jsd=lmho.workspace(lmho.fljsd_bwd_workspace_bytes(Tf, H, Vf)),
                       p0=lmho.workspace(lmho.flce_workspace_bytes(Tf, H, 1000)),
                       p1=lmho.workspace(lmho.flce_workspace_bytes(Tf, H, Vf - 1000)))
        self.Vf = Vf

    def run(self):
        L, o, w = self.lmho, self.out, self.ws
        L.ce_fwd_f32(self.z, self.t, loss=o["ce"], ws=w["ce"])
        L.ce_fwd_sbv_bf16(self.zb, self.tb, loss=o["sbv"])
        L.flce_fwd_bwd_bf16(self.x, self.W, self.tt, 0.5, loss=o["flce"], dx=o["dx"], dW=o["dW"], ws=w["flce"])
        L.fljsd_fwd_bwd_bf16(self.x, self.W, self.xt, self.Wt, 0.4, 1.5, self.keep, 1.0, loss=o["jsd"], dxs=o["dxs"],
                             dWs=o["dWs"], ws=w["jsd"])
        for j, (v0, n) in enumerate(((0, 1000), (1000, self.Vf - 1000))):
            L.flce_partials_bf16(self.x, self.W[v0:v0 + n], self.tt, v0, partials=o["parts"][j],
                                 ws=w["p0" if j == 0 else "p1"])
        L.ce_merge_partials(o["parts"].view(2, 3, -1, 1), self.tt.view(-1, 1), self.Vf, loss=o["vp_rows"].view(-1, 1))
        L.rows_mean(o["vp_rows"], out=o["vp_mean"])

    def results(self):
        torch.cuda.synchronize()
        return {k: v.clone() for k, v in self.out.items()}


def test_step_replays_bitwise_in_a_cuda_graph(gpu_lib):
    s = Step(gpu_lib, 90)
    s.run()                                   # eager: one-time host set-up happens here
    eager = s.results()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        s.run()                               # warm-up on the capture stream's side, as torch recommends
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        s.run()
    for _ in range(3):
        g.replay()
        got = s.results()
        for k in eager:
            assert torch.equal(got[k], eager[k]), k
    # new inputs in the same buffers: the replay follows them
    n = Step(gpu_lib, 91)
    for name in ("z", "t", "zb", "tb", "x", "W", "xt", "Wt", "tt"):
        getattr(s, name).copy_(getattr(n, name))
    n.run()
    fresh = n.results()
    g.replay()
    got = s.results()
    for k in fresh:
        assert torch.equal(got[k], fresh[k]), k
    for k in ("ce", "flce", "jsd", "vp_mean"):
        assert not torch.equal(fresh[k], eager[k]), k
    for w in s.ws.values():
        assert gpu_lib.ws_status(w) == 0
