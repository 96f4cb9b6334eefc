"""Pins for the fp64 attention oracle (no GPU): PyTorch's independent scaled_dot_product_attention
in fp64, and closed forms that a slip in the scores, the mask, the softmax or the value
product would break."""
import numpy as np
import pytest
import torch

from oracle.attention import attention


def rand16(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


def sdpa64(q, k, v, causal=False, mask=None):
    # the scale the library receives is a float32: 1/sqrt(D) rounded to float32
    t = lambda x: torch.from_numpy(x.astype(np.float64))
    scale = float(np.float32(1.0 / np.sqrt(q.shape[-1])))
    return torch.nn.functional.scaled_dot_product_attention(
        t(q), t(k), t(v), attn_mask=None if mask is None else torch.from_numpy(mask),
        is_causal=causal, scale=scale).numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,S,D", [(1, 2, 37, 64), (2, 1, 130, 128), (1, 3, 5, 16)])
def test_matches_torch_sdpa(causal, B, H, S, D):
    rng = np.random.default_rng(S + D)
    q, k, v = rand16(rng, (B, H, S, D)), rand16(rng, (B, H, S, D)), rand16(rng, (B, H, S, D))
    o, lse, o64 = attention(q, k, v, causal=causal, return_lse=True)
    ref = sdpa64(q, k, v, causal=causal)
    assert np.allclose(o64, ref, rtol=1e-12, atol=1e-12)
    assert np.array_equal(o.view(np.uint16), o64.astype(np.float16).view(np.uint16))


def test_causal_with_fewer_queries_than_keys_is_bottom_right_aligned():
    rng = np.random.default_rng(3)
    B, H, Sq, Skv, D = 1, 2, 7, 19, 32
    q, k, v = rand16(rng, (B, H, Sq, D)), rand16(rng, (B, H, Skv, D)), rand16(rng, (B, H, Skv, D))
    _, _, o64 = attention(q, k, v, causal=True, return_lse=True)
    keep = np.arange(Skv)[None, :] <= np.arange(Sq)[:, None] + (Skv - Sq)
    ref = sdpa64(q, k, v, mask=keep)
    assert np.allclose(o64, ref, rtol=1e-12, atol=1e-12)
    # the last query sees every key: same as unmasked attention for that row
    _, _, full = attention(q, k, v, causal=False, return_lse=True)
    assert np.allclose(o64[:, :, -1], full[:, :, -1], rtol=1e-13, atol=1e-13)


def test_identical_keys_give_the_mean_of_values():
    rng = np.random.default_rng(4)
    q = rand16(rng, (1, 2, 9, 64))
    k = np.broadcast_to(rand16(rng, (1, 2, 1, 64)), (1, 2, 23, 64)).copy()
    v = rand16(rng, (1, 2, 23, 64))
    _, _, o64 = attention(q, k, v, return_lse=True)
    assert np.allclose(o64, v.astype(np.float64).mean(axis=2, keepdims=True), rtol=1e-13, atol=1e-14)


def test_single_key_returns_its_value():
    rng = np.random.default_rng(5)
    q, k, v = rand16(rng, (2, 2, 11, 32)), rand16(rng, (2, 2, 1, 32)), rand16(rng, (2, 2, 1, 32))
    o = attention(q, k, v)
    assert np.array_equal(o, np.broadcast_to(v, o.shape))


def test_causal_first_query_sees_only_the_first_key():
    rng = np.random.default_rng(6)
    q, k, v = rand16(rng, (1, 3, 17, 64)), rand16(rng, (1, 3, 17, 64)), rand16(rng, (1, 3, 17, 64))
    o = attention(q, k, v, causal=True)
    assert np.array_equal(o[:, :, 0], v[:, :, 0])


def test_key_permutation_invariance_without_mask():
    rng = np.random.default_rng(7)
    q, k, v = rand16(rng, (1, 2, 13, 64)), rand16(rng, (1, 2, 29, 64)), rand16(rng, (1, 2, 29, 64))
    perm = rng.permutation(29)
    _, _, a = attention(q, k, v, return_lse=True)
    _, _, b = attention(q, k[:, :, perm], v[:, :, perm], return_lse=True)
    assert np.allclose(a, b, rtol=1e-13, atol=1e-14)


def test_rows_without_keys_are_zero():
    rng = np.random.default_rng(8)
    q, k, v = rand16(rng, (1, 1, 10, 16)), rand16(rng, (1, 1, 4, 16)), rand16(rng, (1, 1, 4, 16))
    o, lse, _ = attention(q, k, v, causal=True, return_lse=True)
    # bottom-right alignment: query i keeps keys j <= i - 6, so queries 0..5 keep none
    assert np.all(o[0, 0, :6] == 0) and np.all(np.isneginf(lse[0, 0, :6]))
    assert np.all(np.isfinite(lse[0, 0, 6:]))


def test_sharp_scores_pick_one_value():
    rng = np.random.default_rng(9)
    k = rand16(rng, (1, 1, 8, 64))
    v = rand16(rng, (1, 1, 8, 64))
    q = (k[:, :, 3:4] * 4).astype(np.float16)            # score gap >> 1 after 1/sqrt(64)
    o = attention(q, k, v, scale=4.0)
    assert np.allclose(o[0, 0, 0].astype(np.float64), v[0, 0, 3].astype(np.float64), atol=2e-3)


def test_lse_matches_logsumexp():
    rng = np.random.default_rng(10)
    q, k, v = rand16(rng, (1, 1, 6, 32)), rand16(rng, (1, 1, 12, 32)), rand16(rng, (1, 1, 12, 32))
    _, lse, _ = attention(q, k, v, return_lse=True)
    s = (q.astype(np.float64)[0, 0] @ k.astype(np.float64)[0, 0].T) * float(np.float32(1 / np.sqrt(32)))
    ref = torch.logsumexp(torch.from_numpy(s), dim=-1).numpy()
    assert np.allclose(lse[0, 0], ref, rtol=1e-13, atol=1e-13)
