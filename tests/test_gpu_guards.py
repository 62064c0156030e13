"""Out-of-bounds and unwritten-output checks of every entry point on the GPU
(compute-sanitizer's job, done with guard regions instead).

Each output and each workspace is a view into a larger buffer whose guard
regions before and after hold a canary byte; outputs are pre-filled with NaN.
After the call: the guards are intact (no write outside the declared ranges,
workspace included), every output element was written (no NaN left, all
targets valid), and every input is bitwise unchanged (the pages' "no mutation"
rule).  Shapes are ragged: T, V and H off the tile sizes, with and without V
and H whole 64-element chunks (both forms of the MN-major tensor maps)."""
import math

import numpy as np
import pytest
import torch

import gen
from tests.helpers import to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

G = 4096          # guard bytes on each side (keeps 256-byte alignment of the view)
CANARY = 0xA5


class Guarded:
    def __init__(self):
        self.bufs = []

    def view(self, nbytes, dtype, shape, fill=float("nan")):
        buf = torch.full((G + nbytes + G,), CANARY, dtype=torch.uint8, device="cuda")
        v = buf[G:G + nbytes]
        if dtype is not torch.uint8:
            v = v.view(dtype).view(shape)
            v.fill_(fill)
        self.bufs.append((buf, nbytes))
        return v

    def ws(self, nbytes):
        buf = torch.full((G + nbytes + G,), CANARY, dtype=torch.uint8, device="cuda")
        v = buf[G:G + nbytes]
        v.zero_()
        self.bufs.append((buf, nbytes))
        return v

    def check(self):
        torch.cuda.synchronize()
        for buf, nbytes in self.bufs:
            assert bool((buf[:G] == CANARY).all()), "write before the range"
            assert bool((buf[G + nbytes:] == CANARY).all()), "write past the range"


def snapshot(*ts):
    return [t.clone() for t in ts]


def unchanged(before, after):
    torch.cuda.synchronize()
    for a, b in zip(before, after):
        assert torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.uint8) if b.dtype == torch.bfloat16 else b)


def written(*ts):
    for t in ts:
        assert bool(torch.isfinite(t.float()).all()), "an output element was never written"


@pytest.mark.parametrize("T,V", [(37, 1001), (300, 4096), (5, 70000)])
def test_ce_f32_guards(gpu_lib, T, V):
    g = Guarded()
    z = to_dev(gen.normal_f32(20, 0, (T, V)))
    t = to_dev(gen.targets(20, 1, (T,), V))
    before = snapshot(z, t)
    loss = g.view(4, torch.float32, (1,))
    ws = g.ws(gpu_lib.ce_workspace_bytes(T, V))
    gpu_lib.ce_fwd_f32(z, t, loss=loss, ws=ws)
    g.check()
    written(loss, gpu_lib.row_losses(ws, T))
    unchanged(before, [z, t])
    dl = g.view(4 * T * V, torch.float32, (T, V))
    loss2 = g.view(4, torch.float32, (1,))
    ws2 = g.ws(gpu_lib.ce_workspace_bytes(T, V))
    gpu_lib.ce_fwd_bwd_f32(z, t, 2.0, loss=loss2, dlogits=dl, ws=ws2)
    g.check()
    written(loss2, dl)
    unchanged(before, [z, t])


@pytest.mark.parametrize("S,B,V", [(5, 3, 777), (64, 4, 4096), (3, 2, 40000)])
def test_ce_sbv_guards(gpu_lib, S, B, V):
    g = Guarded()
    z = to_dev_bf16(gen.normal_bf16_bits(21, 0, (S, B, V), sigma=2.0))
    t = to_dev(gen.targets(21, 1, (S, B), V))
    dloss = to_dev(gen.normal_f32(21, 2, (S, B)))
    before = snapshot(z, t, dloss)
    loss = g.view(4 * S * B, torch.float32, (S, B))
    gpu_lib.ce_fwd_sbv_bf16(z, t, loss=loss)
    g.check()
    written(loss)
    loss2 = g.view(4 * S * B, torch.float32, (S, B))
    dl = g.view(2 * S * B * V, torch.bfloat16, (S, B, V))
    gpu_lib.ce_fwd_bwd_sbv_bf16(z, t, dloss=dloss, grad_scale=0.5, loss=loss2, dlogits=dl)
    g.check()
    written(loss2, dl)
    unchanged(before, [z, t, dloss])


FUSED = [(70, 200, 300), (130, 256, 4096), (33, 72, 640), (257, 128, 1000)]


@pytest.mark.parametrize("T,H,V", FUSED)
def test_flce_guards(gpu_lib, T, H, V):
    g = Guarded()
    x = to_dev_bf16(gen.normal_bf16_bits(22, 0, (T, H)))
    W = to_dev_bf16(gen.normal_bf16_bits(22, 2, (V, H), sigma=1.0 / math.sqrt(H)))
    t = to_dev(gen.targets(22, 1, (T,), V))
    before = snapshot(x, W, t)
    loss = g.view(4, torch.float32, (1,))
    ws = g.ws(gpu_lib.flce_workspace_bytes(T, H, V))
    gpu_lib.flce_fwd_bf16(x, W, t, loss=loss, ws=ws)
    g.check()
    assert gpu_lib.ws_status(ws) == 0
    written(loss, gpu_lib.row_losses(ws, T))
    loss2 = g.view(4, torch.float32, (1,))
    dx = g.view(4 * T * H, torch.float32, (T, H))
    dW = g.view(4 * V * H, torch.float32, (V, H))
    ws2 = g.ws(gpu_lib.flce_bwd_workspace_bytes(T, H, V))
    gpu_lib.flce_fwd_bwd_bf16(x, W, t, 3.0, loss=loss2, dx=dx, dW=dW, ws=ws2)
    g.check()
    assert gpu_lib.ws_status(ws2) == 0
    written(loss2, dx, dW)
    unchanged(before, [x, W, t])


@pytest.mark.parametrize("T,H,V", FUSED)
def test_fljsd_guards(gpu_lib, T, H, V):
    g = Guarded()
    xs = to_dev_bf16(gen.normal_bf16_bits(23, 0, (T, H)))
    xt = to_dev_bf16(gen.normal_bf16_bits(23, 3, (T, H)))
    Ws = to_dev_bf16(gen.normal_bf16_bits(23, 2, (V, H), sigma=1.0 / math.sqrt(H)))
    Wt = to_dev_bf16(gen.normal_bf16_bits(23, 4, (V, H), sigma=1.0 / math.sqrt(H)))
    keep = to_dev((gen.targets(23, 1, (T,), 3) != 0).astype(np.uint8))
    before = snapshot(xs, Ws, xt, Wt, keep)
    loss = g.view(4, torch.float32, (1,))
    ws = g.ws(gpu_lib.fljsd_workspace_bytes(T, H, V))
    gpu_lib.fljsd_fwd_bf16_ex(xs, Ws, xt, Wt, 0.3, temperature=1.5, keep=keep, loss=loss, ws=ws)
    g.check()
    assert gpu_lib.ws_status(ws) == 0
    written(loss)
    loss2 = g.view(4, torch.float32, (1,))
    dxs = g.view(4 * T * H, torch.float32, (T, H))
    dWs = g.view(4 * V * H, torch.float32, (V, H))
    ws2 = g.ws(gpu_lib.fljsd_bwd_workspace_bytes(T, H, V))
    gpu_lib.fljsd_fwd_bwd_bf16(xs, Ws, xt, Wt, 0.5, temperature=1.0, keep=keep, grad_scale=2.0, loss=loss2,
                               dxs=dxs, dWs=dWs, ws=ws2)
    g.check()
    assert gpu_lib.ws_status(ws2) == 0
    written(loss2, dxs, dWs)
    unchanged(before, [xs, Ws, xt, Wt, keep])


@pytest.mark.parametrize("B,S,H,V", [(4, 33, 128, 1000), (2, 65, 256, 4096)])
def test_cpo_guards(gpu_lib, B, S, H, V):
    g = Guarded()
    x = to_dev_bf16(gen.normal_bf16_bits(24, 0, (B, S, H)))
    W = to_dev_bf16(gen.normal_bf16_bits(24, 2, (V, H), sigma=1.0 / math.sqrt(H)))
    t = to_dev(gen.targets(24, 1, (B, S), V))
    before = snapshot(x, W, t)
    loss = g.view(4, torch.float32, (1,))
    lp = g.view(4 * B, torch.float32, (B,))
    ws = g.ws(gpu_lib.flce_cpo_workspace_bytes(B, S, H, V))
    gpu_lib.flce_cpo_fwd_bf16(x, W, t, 0.2, 1.0, loss=loss, logps=lp, ws=ws)
    g.check()
    assert gpu_lib.ws_status(ws) == 0
    written(loss, lp)
    loss2 = g.view(4, torch.float32, (1,))
    lp2 = g.view(4 * B, torch.float32, (B,))
    dx = g.view(4 * B * S * H, torch.float32, (B, S, H))
    dW = g.view(4 * V * H, torch.float32, (V, H))
    ws2 = g.ws(gpu_lib.flce_cpo_bwd_workspace_bytes(B, S, H, V))
    gpu_lib.flce_cpo_fwd_bwd_bf16(x, W, t, 0.2, 1.0, 1.0, loss=loss2, logps=lp2, dx=dx, dW=dW, ws=ws2)
    g.check()
    assert gpu_lib.ws_status(ws2) == 0
    written(loss2, lp2, dx, dW)
    unchanged(before, [x, W, t])


@pytest.mark.parametrize("S,B,V,shards", [(7, 3, 1001, 3), (64, 4, 4096, 2), (3, 2, 70000, 8)])
def test_vocab_parallel_guards(gpu_lib, S, B, V, shards):
    """Each shard's partials and the merged losses inside guard regions; the
    shards are separate buffers as on separate ranks (odd widths included)."""
    g = Guarded()
    z = gen.normal_bf16_bits(24, 0, (S, B, V), sigma=2.0)
    t = to_dev(gen.targets(24, 1, (S, B), V))
    cuts = [round(V * j / shards) + (j % 2) for j in range(shards)] + [V]
    cuts[0] = 0
    parts = g.view(shards * 3 * S * B * 4, torch.float32, (shards, 3, S, B))
    locals_ = []
    for j in range(shards):
        v0, w = cuts[j], cuts[j + 1] - cuts[j]
        local = to_dev_bf16(np.ascontiguousarray(z[..., v0:v0 + w]))
        locals_.append(local)
        before = snapshot(local, t)
        gpu_lib.ce_partials_sbv_bf16(local, t, v0, partials=parts[j])
        unchanged(before, [local, t])
    loss = g.view(S * B * 4, torch.float32, (S, B))
    before = snapshot(parts, t)
    gpu_lib.ce_merge_partials(parts, t, V, loss=loss)
    g.check()
    unchanged(before, [parts, t])
    torch.cuda.synchronize()
    assert not bool(torch.isnan(parts).any()), "a partial was never written"   # -inf is a valid target logit
    written(loss)


@pytest.mark.parametrize("T,H,V", FUSED)
def test_vocab_parallel_fused_guards(gpu_lib, T, H, V):
    """The shard calls of the vocab-parallel fused losses on an uneven 2-way
    split of W's rows, and their merges, each into guarded outputs."""
    g = Guarded()
    x = to_dev_bf16(gen.normal_bf16_bits(26, 0, (T, H)))
    xt = to_dev_bf16(gen.normal_bf16_bits(26, 3, (T, H)))
    W = to_dev_bf16(gen.normal_bf16_bits(26, 2, (V, H), sigma=1.0 / math.sqrt(H)))
    Wt = to_dev_bf16(gen.normal_bf16_bits(26, 4, (V, H), sigma=1.0 / math.sqrt(H)))
    t = to_dev(gen.targets(26, 1, (T,), V))
    keep = to_dev((gen.targets(26, 5, (T,), 3) != 0).astype(np.uint8))
    cut = V // 3 if V > 1 else 1
    shards = [(0, cut), (cut, V - cut)] if V > 1 else [(0, 1)]
    before = snapshot(x, xt, W, Wt, t, keep)
    k = len(shards)
    parts = g.view(k * 3 * T * 4, torch.float32, (k, 3, T))
    lparts = g.view(k * 2 * T * 4, torch.float32, (k, 2, T))
    terms = g.view(k * T * 4, torch.float32, (k, T))
    for j, (v0, w) in enumerate(shards):
        ws = g.ws(max(gpu_lib.flce_workspace_bytes(T, H, w), gpu_lib.fljsd_workspace_bytes(T, H, w)))
        gpu_lib.flce_partials_bf16(x, W[v0:v0 + w], t, v0, partials=parts[j], ws=ws)
        gpu_lib.fljsd_lse_partials_bf16(x, W[v0:v0 + w], xt, Wt[v0:v0 + w], 1.5, out=lparts[j], ws=ws)
        g.check()
        assert gpu_lib.ws_status(ws) == 0
    lse = g.view(2 * T * 4, torch.float32, (2, T))
    gpu_lib.lse_merge_partials(lparts, out=lse)
    kls = g.view(k * T * 4, torch.float32, (k, T))
    for j, (v0, w) in enumerate(shards):
        ws = g.ws(gpu_lib.fljsd_workspace_bytes(T, H, w))
        gpu_lib.fljsd_terms_bf16(x, W[v0:v0 + w], xt, Wt[v0:v0 + w], lse, 0.3, 1.5, out=terms[j], ws=ws,
                                 kl_local=kls[j])
        g.check()
        assert gpu_lib.ws_status(ws) == 0
    kl = g.view(T * 4, torch.float32, (T,))
    gpu_lib.jsd_merge_terms(kls, rows=kl, loss=g.view(4, torch.float32, (1,)))
    for v0, w in shards:
        dxs = g.view(4 * T * H, torch.float32, (T, H))
        dWs = g.view(4 * w * H, torch.float32, (w, H))
        ws = g.ws(gpu_lib.fljsd_bwd_workspace_bytes(T, H, w))
        gpu_lib.fljsd_shard_bwd_bf16(x, W[v0:v0 + w], xt, Wt[v0:v0 + w], lse, kl, 0.3, 1.5, keep, 2.0, dx=dxs, dW=dWs,
                                     ws=ws)
        g.check()
        assert gpu_lib.ws_status(ws) == 0
        written(dxs, dWs)
    rows = g.view(T * 4, torch.float32, (T,))
    loss = g.view(4, torch.float32, (1,))
    gpu_lib.jsd_merge_terms(terms, keep, rows=rows, loss=loss)
    ce_rows = g.view(T * 4, torch.float32, (T, 1))
    gpu_lib.ce_merge_partials(parts.view(k, 3, T, 1), t.view(T, 1), V, loss=ce_rows)
    mean = g.view(4, torch.float32, (1,))
    gpu_lib.rows_mean(ce_rows.view(T), out=mean)
    grads = []
    for v0, w in shards:
        dx = g.view(4 * T * H, torch.float32, (T, H))
        dW = g.view(4 * w * H, torch.float32, (w, H))
        ws = g.ws(gpu_lib.flce_bwd_workspace_bytes(T, H, w))
        gpu_lib.flce_shard_bwd_bf16(x, W[v0:v0 + w], t, parts, v0, V, 1.5, dx=dx, dW=dW, ws=ws)
        g.check()
        assert gpu_lib.ws_status(ws) == 0
        grads += [dx, dW]
    g.check()
    assert not bool(torch.isnan(parts).any()), "a partial was never written"   # -inf is a valid target logit
    written(lparts, lse, terms, kls, kl, rows, loss, ce_rows, mean, *grads)
    unchanged(before, [x, xt, W, Wt, t, keep])


def test_vocab_parallel_cpo_guards(gpu_lib):
    """cpo_combine_rows and the weighted shard backward into guarded outputs."""
    g = Guarded()
    B, S, H, V = 4, 33, 200, 640
    T = B * S
    x = to_dev_bf16(gen.normal_bf16_bits(28, 0, (T, H)))
    W = to_dev_bf16(gen.normal_bf16_bits(28, 2, (V, H), sigma=1.0 / math.sqrt(H)))
    t = to_dev(gen.targets(28, 1, (T,), V))
    rows = to_dev(np.abs(gen.normal_f32(28, 3, (T,))) + 1.0)
    before = snapshot(x, W, t, rows)
    loss = g.view(4, torch.float32, (1,))
    logps = g.view(4 * B, torch.float32, (B,))
    row_w = g.view(4 * T, torch.float32, (T,))
    gpu_lib.cpo_combine_rows(rows, B, 0.2, 0.8, loss=loss, logps=logps, row_w=row_w,
                             ws=g.ws(gpu_lib.cpo_combine_workspace_bytes(B)))
    g.check()
    written(loss, logps, row_w)
    parts = torch.empty((2, 3, T), device="cuda")
    shards = [(0, 300), (300, V - 300)]
    for j, (v0, w) in enumerate(shards):
        gpu_lib.flce_partials_bf16(x, W[v0:v0 + w], t, v0, partials=parts[j])
    for v0, w in shards:
        dx = g.view(4 * T * H, torch.float32, (T, H))
        dW = g.view(4 * w * H, torch.float32, (w, H))
        ws = g.ws(gpu_lib.flce_bwd_workspace_bytes(T, H, w))
        gpu_lib.flce_shard_bwd_bf16(x, W[v0:v0 + w], t, parts, v0, V, 1.2, dx=dx, dW=dW, ws=ws, row_w=row_w)
        g.check()
        assert gpu_lib.ws_status(ws) == 0
        written(dx, dW)
    unchanged(before, [x, W, t, rows])


def test_flat_f32_vocab_parallel_guards(gpu_lib):
    g = Guarded()
    T, V = 37, 1001
    z = to_dev(gen.normal_f32(27, 0, (T, V)))
    t = to_dev(gen.targets(27, 1, (T,), V))
    before = snapshot(z, t)
    shards = [(0, 333), (333, V - 333)]
    parts = g.view(2 * 3 * T * 4, torch.float32, (2, 3, T))
    for j, (v0, w) in enumerate(shards):
        gpu_lib.ce_partials_f32(z[:, v0:v0 + w].contiguous(), t, v0, partials=parts[j])
    g.check()
    unchanged(before, [z, t])
    assert not bool(torch.isnan(parts).any()), "a partial was never written"


def test_probe_read_guards(gpu_lib):
    g = Guarded()
    words = gen.targets(25, 0, (5 * 4096,), 2 ** 32).astype(np.uint32)
    data = torch.from_numpy(words.view(np.int32)).cuda()
    out = g.view(5 * 4, torch.int32, (5,), fill=0)
    before = snapshot(data)
    gpu_lib.probe_read(data, 16384, out=out)
    g.check()
    unchanged(before, [data])
    want = np.bitwise_xor.reduce(words.reshape(5, -1), axis=1)
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32), want)
