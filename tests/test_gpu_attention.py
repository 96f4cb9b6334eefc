"""GPU parity of flash_attention_fwd against the fp64 attention oracle.

Acceptance: per element |gpu - oracle| <= 1e-2 + 1e-2 |oracle| (the operator tests' bound),
relative Frobenius error <= 2e-3 (P is rounded to fp16 before the second product: about
2^-12 relative per probability, averaged over the keys), log-sum-exp within 1e-3.
"""
import numpy as np
import pytest
import torch

import tensor_core_gemm_multistage_gb300 as gsr
from oracle.attention import attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    gsr.build()
    yield


def inputs(B, H, Sq, Skv, D, seed, same_keys=False):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, Sq, D, generator=g).half()
    k = torch.randn(B, H, Skv, D, generator=g).half()
    if same_keys:
        k = k[:, :, :1].expand(B, H, Skv, D).contiguous()
    v = torch.randn(B, H, Skv, D, generator=g).half()
    return q, k, v


def run(q, k, v, causal=False, scale=0.0):
    dev = torch.device("cuda", 0)
    B, H, Sq, D = q.shape
    O = torch.full((B, H, Sq, D), float("nan"), dtype=torch.float16, device=dev)
    lse = torch.full((B, H, Sq), float("nan"), dtype=torch.float32, device=dev)
    gsr.flash_attention_fwd(q.to(dev), k.to(dev), v.to(dev), O, lse, softmax_scale=scale, causal=causal)
    status, code = gsr.device_status()
    assert status == gsr.Status.OK, hex(code)
    return O.cpu().numpy(), lse.cpu().numpy()


def check(q, k, v, causal=False, scale=0.0):
    o, lse = run(q, k, v, causal, scale)
    ref, ref_lse, _ = attention(q, k, v, scale=None if scale == 0.0 else scale, causal=causal,
                                return_lse=True)
    x = o.astype(np.float64)
    y = ref.astype(np.float64)
    assert not np.isnan(x).any(), "unwritten outputs"
    err = np.abs(x - y)
    assert np.all(err <= 1e-2 + 1e-2 * np.abs(y)), "worst %g" % err.max()
    ny = np.linalg.norm(y)
    if ny > 0:
        assert np.linalg.norm(x - y) / ny <= 2e-3, np.linalg.norm(x - y) / ny
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.all(np.abs(lse[fin] - ref_lse[fin]) <= 1e-3)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,S,D", [(1, 1, 128, 64), (1, 2, 256, 128), (2, 3, 200, 64),
                                     (1, 2, 333, 128), (1, 1, 1024, 128)])
def test_self_attention(B, H, S, D, causal):
    check(*inputs(B, H, S, S, D, seed=S + D), causal=causal)


@pytest.mark.parametrize("Sq,Skv", [(100, 333), (1, 515), (256, 64), (64, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_cross_lengths(Sq, Skv, causal):
    check(*inputs(1, 2, Sq, Skv, 128, seed=Sq * 7 + Skv), causal=causal)


def test_explicit_scale_and_identical_keys():
    q, k, v = inputs(1, 2, 130, 257, 64, seed=3, same_keys=True)
    check(q, k, v, scale=0.3)
    o, _ = run(q, k, v, scale=0.3)
    mean = v.double().mean(dim=2, keepdim=True).numpy()
    assert np.allclose(o.astype(np.float64), np.broadcast_to(mean, o.shape), atol=2e-3)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_negative_scale(D, causal):
    # a negative scale turns the row maximum of the scaled scores into the minimum of the raw ones
    check(*inputs(1, 2, 300, 300, D, seed=11 + D), causal=causal, scale=-0.2)


@pytest.mark.parametrize("causal", [False, True])
def test_peaked_rows(causal):
    # large scores: each row's weight sits on a few keys, often in only one of a tile's key halves
    check(*inputs(2, 1, 384, 384, 128, seed=12), causal=causal, scale=1.5)


def test_no_keys_and_fully_masked_rows():
    q, k, v = inputs(1, 1, 200, 70, 64, seed=4)
    check(q, k, v, causal=True)                    # rows 0..129 have no key
    o, lse = run(q, k, v, causal=True)
    assert np.all(o[0, 0, :130] == 0) and np.all(np.isneginf(lse[0, 0, :130]))
    dev = torch.device("cuda", 0)
    O = torch.full((1, 1, 5, 64), float("nan"), dtype=torch.float16, device=dev)
    lse0 = torch.zeros(1, 1, 5, dtype=torch.float32, device=dev)
    empty = torch.empty(1, 1, 0, 64, dtype=torch.float16, device=dev)
    gsr.flash_attention_fwd(q[:, :, :5].to(dev).contiguous(), empty, empty, O, lse0)
    torch.cuda.synchronize()
    assert torch.all(O == 0) and torch.all(torch.isinf(lse0))


def test_timeout_reports_and_recovers():
    q, k, v = inputs(1, 1, 256, 256, 64, seed=5)
    gsr.set_wait_timeout_ns(50_000_000)
    gsr.set_test_flags(1)
    try:
        dev = torch.device("cuda", 0)
        O = torch.zeros(1, 1, 256, 64, dtype=torch.float16, device=dev)
        gsr.flash_attention_fwd(q.to(dev), k.to(dev), v.to(dev), O)
        status, code = gsr.device_status()
    finally:
        gsr.set_test_flags(0)
        gsr.set_wait_timeout_ns(1_000_000_000)
    assert status == gsr.Status.ERR_DEVICE_TIMEOUT and code & 0xF00 == 0x300
    check(q, k, v)


def test_validation():
    dev = torch.device("cuda", 0)
    t = torch.empty(1, 1, 128, 64, dtype=torch.float16, device=dev)
    L = gsr.lib()
    import ctypes
    vp = ctypes.c_void_p
    args = lambda o, d: (vp(t.data_ptr()), vp(t.data_ptr()), vp(t.data_ptr()), vp(o), None, 1, 1, 128,
                         128, d, ctypes.c_float(0.0), 0, None)
    assert L.flash_attention_fwd(*args(t.data_ptr(), 96)) == gsr.Status.ERR_INVALID_ARG
    assert L.flash_attention_fwd(*args(t.data_ptr(), 64)) == gsr.Status.ERR_ALIAS


# Many work items per CTA: the kernel runs one persistent CTA per SM (152 on GB300), each taking
# (two query tiles, batch x head) items from a device counter one after another, with one item's
# last products overlapping the next item's first.  These shapes have 2-3 items per CTA.
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,S,D", [(4, 40, 512, 64), (2, 80, 700, 128), (3, 33, 1280, 128)])
def test_many_items_per_cta(B, H, S, D, causal):
    check(*inputs(B, H, S, S, D, seed=B * H + S + D), causal=causal)


@pytest.mark.parametrize("Sq,Skv,D", [(1024, 300, 128), (900, 1300, 64)])
def test_many_items_with_keyless_items_between(Sq, Skv, D):
    # causal with Sq > Skv: the first query blocks of every head have no key at all (O = 0,
    # lse = -inf), so items without work sit between items with work in every CTA's sequence
    check(*inputs(2, 100, Sq, Skv, D, seed=Sq + Skv), causal=True)


@pytest.mark.parametrize("causal", [False, True])
def test_bench_workload_sampled_heads(causal):
    # The benchmarked attention workload in full (4 x 32 heads, 4096 x 4096, D 128; 2048 items on
    # 152 CTAs), checked on a sample of heads against the oracle.
    from tensor_core_gemm_multistage_gb300.workloads import ATTN_WORKLOADS, attention_inputs
    w = ATTN_WORKLOADS["attn_b4_h32_s4096_d128"]
    q, k, v = attention_inputs(w, seed=0)
    o, lse = run(q, k, v, causal=causal)
    for b, h in ((0, 0), (1, 17), (3, 31)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref, ref_lse, _ = attention(q[sl], k[sl], v[sl], causal=causal, return_lse=True)
        x = o[sl].astype(np.float64)
        y = ref.astype(np.float64)
        assert not np.isnan(x).any()
        assert np.all(np.abs(x - y) <= 1e-2 + 1e-2 * np.abs(y)), (b, h)
        assert np.linalg.norm(x - y) / np.linalg.norm(y) <= 2e-3, (b, h)
        assert np.all(np.abs(lse[sl] - ref_lse) <= 1e-3), (b, h)


def test_two_streams_at_once_keep_their_own_work_counters():
    # Each stream has its own item counter: two persistent launches running at the same time on
    # two streams must each process exactly their own items, call after call.
    dev = torch.device("cuda", 0)
    cases = [inputs(2, 60, 640, 640, 128, seed=41), inputs(3, 50, 512, 700, 64, seed=42)]
    dq = [tuple(t.to(dev) for t in c) for c in cases]
    outs = [torch.full(c[0].shape, float("nan"), dtype=torch.float16, device=dev) for c in cases]
    streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    torch.cuda.synchronize()
    for _ in range(3):
        for (q, k, v), o, s, causal in zip(dq, outs, streams, (True, False)):
            with torch.cuda.stream(s):
                gsr.flash_attention_fwd(q, k, v, o, causal=causal, stream=s)
    for s in streams:
        assert gsr.device_status(s)[0] == gsr.Status.OK
    for (q, k, v), o, causal in zip(cases, outs, (True, False)):
        ref = attention(q, k, v, causal=causal).astype(np.float64)
        x = o.cpu().numpy().astype(np.float64)
        assert not np.isnan(x).any()
        assert np.all(np.abs(x - ref) <= 1e-2 + 1e-2 * np.abs(ref))


def _random_attention_cases(n, seed):
    # seeded (B, H, Sq, Skv, D, causal, scale): ragged lengths on both sides, Sq above and below
    # Skv (causal diagonals offset either way), both head sizes, default and explicit scales
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 5))
        Sq, Skv = int(rng.integers(1, 700)), int(rng.integers(1, 900))
        D = int(rng.choice([64, 128]))
        out.append((B, H, Sq, Skv, D, bool(rng.integers(0, 2)), float(rng.choice([0.0, 0.05, 0.2]))))
    return out


@pytest.mark.parametrize("B,H,Sq,Skv,D,causal,scale", _random_attention_cases(16, 2028))
def test_random_attention_cases(B, H, Sq, Skv, D, causal, scale):
    check(*inputs(B, H, Sq, Skv, D, seed=B + H + Sq + Skv + D), causal=causal, scale=scale)
