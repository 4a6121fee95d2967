"""Experts in host memory with a device-memory cache of expert slots
(moe_cache_*): results must be bit-identical to the layer with every expert
resident in device memory."""
import numpy as np
import pytest
import torch

import workloads as W
from fp8_routed_expert_gb300 import C, ExpertCache, MoEError
from harness import DeviceWeights, check_output, make_layer, reference, x_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.fixture(scope="module")
def olmoe():
    fam = W.family("olmoe_decode")
    w = W.make_weights(fam)
    return fam, w, DeviceWeights(w), torch.from_numpy(w.w13), torch.from_numpy(w.w2)


def _x(fam, T, seed):
    return W.normal_bf16(seed, W.configs.TID_X, (T, fam.hidden))


def _plain(layer, xb, dw, k):
    out = layer.forward(x_dev(xb), *dw.args(), k)
    torch.cuda.synchronize()
    return out.view(torch.int16).cpu().numpy()


def _cached(cache, xb, dw, k):
    out = cache.forward(x_dev(xb), dw.router_w, dw.router_bias, dw.s13, dw.s2, k)
    torch.cuda.synchronize()
    return out.view(torch.int16).cpu().numpy()


@pytest.mark.parametrize("T,slots", [(1, 16), (8, 56)])
def test_cached_forward_is_bit_identical(olmoe, T, slots):
    fam, w, dw, w13h, w2h = olmoe
    k = fam.top_k
    layer = make_layer(fam, T)
    plain = make_layer(fam, T)
    cache = ExpertCache(layer, w13h, w2h, slots)
    n_active = 0
    for step in range(6):  # new tokens every step: misses, hits and evictions
        xb = _x(fam, T, 7000 + step)
        got = _cached(cache, xb, dw, k)
        assert np.array_equal(got, _plain(plain, xb, dw, k)), f"step {step}"
        n_active += int((layer.routing(T, k)["counts"] > 0).sum().item())
    st = cache.stats()
    assert st["hits"] + st["misses"] == n_active
    assert st["misses"] >= min(n_active, slots) and st["evictions"] > 0
    assert st["bytes_copied"] == st["misses"] * 3 * fam.hidden * fam.inter
    res = cache.resident()
    assert sum(s >= 0 for s in res) == slots
    ref = reference(xb, w, k)
    check_output(got.astype(np.uint16), ref)
    cache.close()


def test_guessed_prefetch_is_used(olmoe):
    """Guessing with the router of the batch itself names exactly its
    experts: after the prefetch the forward copies nothing more."""
    fam, w, dw, w13h, w2h = olmoe
    k, T = fam.top_k, 1
    layer = make_layer(fam, T)
    cache = ExpertCache(layer, w13h, w2h, 16)
    xb = _x(fam, T, 8100)
    xt = x_dev(xb)
    guess = cache.guess(xt, dw.router_w, dw.router_bias, k, 8)
    assert len(guess) == k and len(set(guess)) == k
    assert cache.prefetch(guess) == k
    before = cache.stats()
    out = _cached(cache, xb, dw, k)
    after = cache.stats()
    assert after["misses"] == before["misses"] and after["prefetch_used"] == k
    active = np.nonzero(layer.routing(T, k)["counts"].cpu().numpy())[0].tolist()
    assert sorted(guess) == active
    assert np.array_equal(out, _plain(make_layer(fam, T), xb, dw, k))
    cache.close()


def test_prefill_batch_through_the_cache(olmoe):
    """The grouped-GEMM path (T > 64) on the cached range."""
    fam, w, dw, w13h, w2h = olmoe
    k, T = fam.top_k, 300
    layer = make_layer(fam, T)
    cache = ExpertCache(layer, w13h, w2h, fam.n_experts)
    xb = _x(fam, T, 8200)
    assert np.array_equal(_cached(cache, xb, dw, k), _plain(make_layer(fam, T), xb, dw, k))
    cache.close()


def test_cache_limits(olmoe):
    fam, w, dw, w13h, w2h = olmoe
    layer = make_layer(fam, 8)
    with pytest.raises(MoEError) as e:
        ExpertCache(layer, w13h, w2h, fam.n_experts + 1)
    assert e.value.code == C["MOE_ERR_SHAPE"]
    cache = ExpertCache(layer, w13h, w2h, 4)
    with pytest.raises(MoEError) as e:   # 8 tokens x top-8 need more than 4 slots
        _cached(cache, _x(fam, 8, 8300), dw, fam.top_k)
    assert e.value.code == C["MOE_ERR_NOMEM"]
    cache.close()


def test_tiny_layer_and_gemv_path_through_the_cache():
    """Small experts (64 KiB of W13) and the GEMV fallback path."""
    fam = W.family("tiny")
    w = W.make_weights(fam)
    dw = DeviceWeights(w)
    for path in ("auto", "gemv"):
        layer = make_layer(fam, 2)   # 2 tokens x top-2: at most 4 experts per batch
        layer.set_path(path)
        plain = make_layer(fam, 2)
        plain.set_path(path)
        cache = ExpertCache(layer, torch.from_numpy(w.w13), torch.from_numpy(w.w2), 4)
        for step in range(6):
            xb = _x(fam, 2, 8400 + step)
            assert np.array_equal(_cached(cache, xb, dw, fam.top_k), _plain(plain, xb, dw, fam.top_k))
        cache.close()
