"""GPU parity of the cross-entropy kernels against the fp64 oracle.

Pages "Cross-entropy loss" (fp32 [tokens, vocab] logits, int64 targets, mean
loss[1]) and "Vocab-parallel cross-entropy, Megatron layout" (bf16 [seq,
batch, vocab], per-token fp32 losses).  Tolerances: fp32 losses relative
1e-5 (per token and mean; a 1e-6 absolute floor covers losses that are ~0,
where the fp32 exp/log of the online normaliser leaves ~1e-7); bf16 logits
accumulated in fp32: absolute 2e-3 per token.
"""
import math

import numpy as np
import pytest
import torch

import gen
import oracle
from tests.helpers import rows_bf16, rows_f32, sample_rows, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

RTOL_F32, ATOL_F32 = 1e-5, 1e-6
ATOL_BF16 = 2e-3
VARIANTS = ["auto", "warp", "cta", "cta512", "cluster2", "cluster4", "cluster8", "bulk"]


@pytest.fixture(autouse=True)
def _auto_variant(gpu_lib):
    gpu_lib.set_ce_variant("auto")
    yield
    gpu_lib.set_ce_variant("auto")


def run_flat(lmho, z, t, ws_extra=0):
    zd, td = to_dev(z), to_dev(t)
    ws = lmho.workspace(lmho.ce_workspace_bytes(*z.shape) + ws_extra)
    loss = lmho.ce_fwd_f32(zd, td, ws=ws)
    torch.cuda.synchronize()
    return float(loss.item()), lmho.row_losses(ws, z.shape[0]).cpu().numpy().astype(np.float64)


# ---------------------------------------------------------------- flat fp32
# The last three put tens of rows on every persistent CTA, so ring stages and
# barriers are reused many times over.
FLAT_SHAPES = [(1, 1), (3, 1), (7, 2), (5, 3), (9, 5), (4, 8), (33, 4095), (17, 4097), (64, 4096),
               (3, 131071), (130, 8192), (5, 65537), (300, 1000), (9000, 1024), (3000, 8192), (700, 24576)]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("T,V", FLAT_SHAPES)
def test_flat_f32_matches_oracle(gpu_lib, variant, T, V):
    gpu_lib.set_ce_variant(variant)
    z = gen.normal_f32(1, 0, (T, V))
    t = gen.targets(1, 1, (T,), V)
    m, rows = run_flat(gpu_lib, z, t)
    m_ref, rows_ref = oracle.ce_f32(z, t)
    np.testing.assert_allclose(rows, rows_ref, rtol=RTOL_F32, atol=ATOL_F32)
    assert m == pytest.approx(m_ref, rel=RTOL_F32, abs=ATOL_F32)


@pytest.mark.parametrize("variant", ["warp", "cta", "cluster4", "bulk"])
def test_flat_unaligned_rows(gpu_lib, variant):
    # logits start 4 bytes past a 16-byte boundary and V*4 is not a multiple of 16:
    # every row has a scalar head and tail around its vector body
    gpu_lib.set_ce_variant(variant)
    T, V = 37, 1001
    z = gen.normal_f32(2, 0, (T * V + 1,))
    t = gen.targets(2, 1, (T,), V)
    zd = to_dev(z)[1:].view(T, V)
    ws = gpu_lib.workspace(gpu_lib.ce_workspace_bytes(T, V))
    loss = gpu_lib.ce_fwd_f32(zd, to_dev(t), ws=ws)
    m_ref, rows_ref = oracle.ce_f32(z[1:].reshape(T, V), t)
    np.testing.assert_allclose(gpu_lib.row_losses(ws, T).cpu().numpy(), rows_ref, rtol=RTOL_F32, atol=ATOL_F32)
    assert float(loss.item()) == pytest.approx(m_ref, rel=RTOL_F32)


EDGE_VARIANTS = ["warp", "cta", "cluster4", "bulk"]


def edge_targets(V):
    # first and last elements, the scalar head and tail of an unaligned row,
    # both sides of 16-byte vector boundaries, the middle; then out of range
    pos = [0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 15, 16, 17, V // 2, V - 17, V - 16, V - 9, V - 8, V - 7, V - 5, V - 4,
           V - 3, V - 2, V - 1]
    return np.array(pos + pos[::-1] + [-1, V], np.int64)


@pytest.mark.parametrize("variant", EDGE_VARIANTS)
def test_flat_targets_at_row_edges(gpu_lib, variant):
    """The target logit is found wherever it sits in the row: in the scalar
    head or tail around the 16-byte vector body, on a vector boundary, first
    or last; an out-of-range target gives NaN for its row only."""
    gpu_lib.set_ce_variant(variant)
    V = 1001
    t = edge_targets(V)
    T = len(t)
    z = gen.normal_f32(12, 0, (T * V + 1,), sigma=3.0)
    zd = to_dev(z)[1:].view(T, V)      # 4 bytes past a 16-byte boundary
    ws = gpu_lib.workspace(gpu_lib.ce_workspace_bytes(T, V))
    gpu_lib.ce_fwd_f32(zd, to_dev(t), ws=ws)
    rows = gpu_lib.row_losses(ws, T).cpu().numpy().astype(np.float64)
    ok = (t >= 0) & (t < V)
    _, rows_ref = oracle.ce_f32(z[1:].reshape(T, V)[ok], t[ok])
    np.testing.assert_allclose(rows[ok], rows_ref, rtol=RTOL_F32, atol=ATOL_F32)
    assert np.all(np.isnan(rows[~ok]))


@pytest.mark.parametrize("variant", EDGE_VARIANTS)
def test_sbv_targets_at_row_edges(gpu_lib, variant):
    # odd V: consecutive bf16 rows start at every 2-byte offset of a 16-byte vector
    gpu_lib.set_ce_variant(variant)
    V = 1001
    t = edge_targets(V)
    S = len(t) // 2
    z = gen.normal_bf16_bits(13, 0, (S, 2, V), sigma=3.0)
    got = run_sbv(gpu_lib, z, t.reshape(S, 2)).reshape(-1)
    ok = (t >= 0) & (t < V)
    want = oracle.ce_sbv_bf16(z.reshape(1, S * 2, V)[:, ok], t[ok].reshape(1, -1)).reshape(-1)
    np.testing.assert_allclose(got[ok], want, rtol=0, atol=ATOL_BF16)
    assert np.all(np.isnan(got[~ok]))


def test_flat_equal_logits_and_shift(gpu_lib):
    T, V = 8, 5000
    z = np.full((T, V), 3.0, np.float32)
    m, rows = run_flat(gpu_lib, z, gen.targets(3, 1, (T,), V))
    np.testing.assert_allclose(rows, math.log(V), rtol=RTOL_F32)
    # shift by a power of two on a grid of multiples of 1/8: exact in fp32
    g = np.round(gen.normal_f32(3, 0, (T, V)) * 8) / 8
    t = gen.targets(3, 1, (T,), V)
    _, r0 = run_flat(gpu_lib, g.astype(np.float32), t)
    _, r1 = run_flat(gpu_lib, (g + 64.0).astype(np.float32), t)
    np.testing.assert_allclose(r1, r0, rtol=0, atol=1e-4)


def test_flat_bad_targets_and_nonfinite_give_nan(gpu_lib):
    T, V = 6, 300
    z = gen.normal_f32(4, 0, (T, V))
    z[2, 17] = np.nan
    z[3, 5] = np.inf
    t = gen.targets(4, 1, (T,), V)
    t[0], t[1] = -1, V
    m, rows = run_flat(gpu_lib, z, t)
    assert np.all(np.isnan(rows[:4])) and np.all(np.isfinite(rows[4:]))
    assert math.isnan(m)


def test_flat_deterministic_and_reusable_workspace(gpu_lib):
    T, V = 1000, 3000
    z = to_dev(gen.normal_f32(5, 0, (T, V)))
    t = to_dev(gen.targets(5, 1, (T,), V))
    ws = gpu_lib.workspace(gpu_lib.ce_workspace_bytes(T, V))
    outs = []
    for variant in ("warp", "cta", "cluster2", "bulk"):
        gpu_lib.set_ce_variant(variant)
        for _ in range(5):
            outs.append(gpu_lib.ce_fwd_f32(z, t, ws=ws).clone())
        first = outs[-5]
        for o in outs[-4:]:
            assert torch.equal(o, first)   # bitwise, same workspace reused
    # the ticket word of the workspace is back at zero after every call
    assert int(ws[-256:].view(torch.int32)[1].item()) == 0


def test_flat_full_size_config(gpu_lib):
    """logits fp32 [16384, 4096] ~ N(0,1), seed 0: full mean against the
    oracle run over every row."""
    T, V = 16384, 4096
    z = gen.normal_f32(0, gen.STREAM_LOGITS, (T, V))
    t = gen.targets(0, gen.STREAM_TARGET, (T,), V)
    m, rows = run_flat(gpu_lib, z, t)
    m_ref, rows_ref = oracle.ce_f32(z, t)
    np.testing.assert_allclose(rows, rows_ref, rtol=RTOL_F32, atol=ATOL_F32)
    assert m == pytest.approx(m_ref, rel=RTOL_F32)


@pytest.mark.parametrize("V", [8192, 131072])
def test_flat_vocab_sweep_full_size_sampled(gpu_lib, V):
    """[16384, V] fp32 at full size; 48 sampled rows recomputed on the host."""
    T = 16384
    z = gen.normal_f32(0, gen.STREAM_LOGITS, (T, V))
    t = gen.targets(0, gen.STREAM_TARGET, (T,), V)
    m, rows = run_flat(gpu_lib, z, t)
    idx = sample_rows(T, 48)
    _, rows_ref = oracle.ce_f32(z[idx], t[idx])
    np.testing.assert_allclose(rows[idx], rows_ref, rtol=RTOL_F32, atol=ATOL_F32)
    # the mean is the fp64 mean of the kernel's own per-token losses
    assert m == pytest.approx(rows.mean(), rel=1e-6)
    assert abs(m - (math.log(V) + 0.5)) < 0.05


# ---------------------------------------------------------------- Megatron bf16
def run_sbv(lmho, z_bits, t):
    out = lmho.ce_fwd_sbv_bf16(to_dev_bf16(z_bits), to_dev(t))
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


SBV_SHAPES = [(1, 1, 1), (3, 2, 5), (7, 3, 4095), (16, 4, 8193), (2, 4, 32768), (3, 1, 131072), (33, 4, 1000),
              (2048, 4, 2048), (700, 4, 16384)]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("S,B,V", SBV_SHAPES)
def test_sbv_bf16_matches_oracle(gpu_lib, variant, S, B, V):
    gpu_lib.set_ce_variant(variant)
    z = gen.normal_bf16_bits(6, 0, (S, B, V), sigma=2.0)
    t = gen.targets(6, 1, (S, B), V)
    got = run_sbv(gpu_lib, z, t)
    np.testing.assert_allclose(got, oracle.ce_sbv_bf16(z, t), rtol=0, atol=ATOL_BF16)


def test_sbv_layout_and_closed_form(gpu_lib):
    S, B, V = 4, 3, 64
    z = np.zeros((S, B, V), np.float32)
    t = np.zeros((S, B), np.int64)
    for s in range(S):
        for b in range(B):
            z[s, b, (s + 2 * b) % V] = 1 + s * B + b
            t[s, b] = (s + 2 * b + 1) % V
    bits = (z.view(np.uint32) >> 16).astype(np.uint16)
    got = run_sbv(gpu_lib, bits, t)
    want = np.log(V - 1 + np.exp(1.0 + np.arange(S * B).reshape(S, B)))
    np.testing.assert_allclose(got, want, rtol=0, atol=ATOL_BF16)


@pytest.mark.parametrize("V", [4096, 131072])
def test_sbv_full_size_sampled(gpu_lib, V):
    """bf16 [2048, 4, V] ~ N(0, 2^2): sampled tokens against the oracle."""
    S, B = 2048, 4
    z = gen.normal_bf16_bits(0, gen.STREAM_LOGITS, (S, B, V), sigma=2.0)
    t = gen.targets(0, gen.STREAM_TARGET, (S, B), V)
    got = run_sbv(gpu_lib, z, t).reshape(-1)
    idx = sample_rows(S * B, 64)
    ref = oracle.ce_sbv_bf16(z.reshape(S * B, 1, V)[idx], t.reshape(-1, 1)[idx]).reshape(-1)
    np.testing.assert_allclose(got[idx], ref, rtol=0, atol=ATOL_BF16)
    assert np.all(np.isfinite(got))


def test_sbv_all_configs_sampled_rows_from_generator(gpu_lib):
    """Each Megatron vocab of the workload table at full [2048, 4, V]: rows
    regenerated on the host by counter offset (not copied back from the GPU)."""
    S, B = 2048, 4
    for V in (8192, 16384, 32768, 65536):
        z = gen.normal_bf16_bits(0, gen.STREAM_LOGITS, (S, B, V), sigma=2.0)
        t = gen.targets(0, gen.STREAM_TARGET, (S, B), V)
        got = run_sbv(gpu_lib, z, t).reshape(-1)
        del z
        idx = sample_rows(S * B, 16, seed=V)
        host_rows = rows_bf16(0, gen.STREAM_LOGITS, idx, V, sigma=2.0)
        ref = oracle.ce_sbv_bf16(host_rows.reshape(len(idx), 1, V), t.reshape(-1, 1)[idx]).reshape(-1)
        np.testing.assert_allclose(got[idx], ref, rtol=0, atol=ATOL_BF16)


def test_flat_rows_regenerated_by_offset(gpu_lib):
    T, V = 4096, 16384
    z = gen.normal_f32(0, 0, (T, V))
    t = gen.targets(0, 1, (T,), V)
    _, rows = run_flat(gpu_lib, z, t)
    idx = sample_rows(T, 8, seed=1)
    _, ref = oracle.ce_f32(rows_f32(0, 0, idx, V), t[idx])
    np.testing.assert_allclose(rows[idx], ref, rtol=RTOL_F32, atol=ATOL_F32)


def test_api_errors_raise(gpu_lib):
    z = torch.zeros((4, 8), device="cuda")
    t = torch.zeros(4, dtype=torch.int64, device="cuda")
    ws = gpu_lib.workspace(gpu_lib.ce_workspace_bytes(4, 8))
    with pytest.raises(gpu_lib.LmhoError) as e:
        gpu_lib.ce_fwd_f32(z, t, loss=z.view(-1)[:1], ws=ws)   # loss aliases logits
    assert e.value.status == gpu_lib.LMHO_ERR_ALIAS
    with pytest.raises(gpu_lib.LmhoError) as e:
        gpu_lib.ce_fwd_f32(z, t, ws=ws[:64])
    assert e.value.status == gpu_lib.LMHO_ERR_WORKSPACE
    with pytest.raises(TypeError):
        gpu_lib.ce_fwd_f32(z.double(), t)


def test_launch_events_are_per_host_thread(gpu_lib):
    """lmho_set_launch_events applies to the calls of the thread that set it:
    another thread's call, queued behind a sleeping kernel on its own stream,
    leaves this thread's events alone (were they recorded there, they would
    still be pending); this thread's next call records them."""
    import threading
    z = to_dev_bf16(gen.normal_bf16_bits(5, 0, (16, 4, 512), sigma=2.0))
    t = to_dev(gen.targets(5, 1, (16, 4), 512))
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    for e in evs:
        e.record()
    torch.cuda.synchronize()
    gpu_lib.set_launch_events(evs)
    side = torch.cuda.Stream()

    def other():
        with torch.cuda.stream(side):
            torch.cuda._sleep(100_000_000)          # tens of milliseconds of GPU time
            gpu_lib.ce_fwd_sbv_bf16(z, t, stream=side)

    th = threading.Thread(target=other)
    th.start()
    th.join()
    try:
        assert all(e.query() for e in evs), "another thread's call recorded this thread's events"
        gpu_lib.ce_fwd_sbv_bf16(z, t)
    finally:
        gpu_lib.set_launch_events(None)
    torch.cuda.synchronize()
    assert evs[0].elapsed_time(evs[1]) > 0.0


@pytest.mark.parametrize("variant", ["auto", "warp", "cta", "cluster2"])
def test_back_to_back_calls_equal_separate_calls(gpu_lib, variant):
    # The row kernels are launched as programmatic dependents of the kernel
    # before them, so queued calls overlap one call's drain with the next one's
    # block launch.  Calls queued without synchronisation -- flat calls sharing
    # one workspace, Megatron calls on alternating inputs -- must give exactly
    # the results of the same calls made one at a time.
    gpu_lib.set_ce_variant(variant)
    try:
        zs = [to_dev(gen.normal_f32(80 + k, 0, (512, 4096))) for k in range(2)]
        ts = [to_dev(gen.targets(80 + k, 1, (512,), 4096)) for k in range(2)]
        zb = [to_dev_bf16(gen.normal_bf16_bits(82 + k, 0, (64, 4, 4096), sigma=2.0)) for k in range(2)]
        tb = [to_dev(gen.targets(82 + k, 1, (64, 4), 4096)) for k in range(2)]
        ws = gpu_lib.workspace(gpu_lib.ce_workspace_bytes(512, 4096))
        alone_f, alone_b = [], []
        for k in range(2):
            alone_f.append(gpu_lib.ce_fwd_f32(zs[k], ts[k], ws=ws).clone())
            alone_b.append(gpu_lib.ce_fwd_sbv_bf16(zb[k], tb[k]).clone())
            torch.cuda.synchronize()
        n = 12
        out_f = torch.full((n,), float("nan"), device="cuda")
        out_b = torch.full((n, 64, 4), float("nan"), device="cuda")
        for i in range(n):
            gpu_lib.ce_fwd_f32(zs[i % 2], ts[i % 2], loss=out_f[i:i + 1], ws=ws)
            gpu_lib.ce_fwd_sbv_bf16(zb[i % 2], tb[i % 2], loss=out_b[i])
        torch.cuda.synchronize()
        for i in range(n):
            assert torch.equal(out_f[i:i + 1], alone_f[i % 2]), i
            assert torch.equal(out_b[i], alone_b[i % 2]), i
        assert gpu_lib.ws_status(ws) == 0
    finally:
        gpu_lib.set_ce_variant("auto")
