"""CUDA path vs the f64 CPU oracle, through the C ABI (needs an sm_103a GPU)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from fp8_routed_expert_gb300 import C, MoEError
from harness import (DeviceWeights, check_expert_y, check_output, check_routing, gpu_y,
                     make_layer, oracle_expert_y, reference, reference_threaded, run,
                     tile_class_experts, x_dev)
from host_ref import combine_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


_weights = {}


def weights(name):
    if name not in _weights:
        fam = W.family(name)
        w = W.make_weights(fam)
        _weights.clear()
        torch.cuda.empty_cache()
        _weights[name] = (fam, w, DeviceWeights(w))
    return _weights[name]


# ------------------------------------------------------------------ full parity

@pytest.mark.parametrize("path", ["gemv", "gemm", "tcgemv"])
def test_tiny(path):
    fam, w, dw = weights("tiny")
    x = W.make_x(fam, 4)
    layer = make_layer(fam, 4)
    out, r = run(layer, x, dw, fam.top_k, path)
    ref = reference(x, w, fam.top_k)
    check_routing(r, ref, fam.n_experts)
    check_output(out, ref)


@pytest.mark.parametrize("T", [1, 8])
@pytest.mark.parametrize("path", ["gemv", "gemm", "tcgemv"])
def test_olmoe_decode(T, path):
    fam, w, dw = weights("olmoe_decode")
    x = W.make_x(fam, T)
    layer = make_layer(fam, T)
    out, r = run(layer, x, dw, fam.top_k, path)
    ref = reference(x, w, fam.top_k)
    check_routing(r, ref, fam.n_experts)
    check_output(out, ref)


@pytest.mark.parametrize("T", [2, 17, 64, 65, 127, 129, 300, 513])
def test_olmoe_ragged_batches(T):
    """Batches that straddle the GEMV/GEMM switch and the 128-row tiles; T =
    513 (4104 pairs) also the one-CTA / many-CTA switch of the pair sort, with
    a last chunk of 8 pairs."""
    fam, w, dw = weights("olmoe_decode")
    x = W.make_x(fam, T)
    layer = make_layer(fam, T)
    out, r = run(layer, x, dw, fam.top_k, "auto")
    ref = reference(x, w, fam.top_k)
    check_routing(r, ref, fam.n_experts)
    check_output(out, ref)


@pytest.mark.parametrize("T", [2, 17, 65, 300])
def test_tcgemv_ragged_batches(T):
    """Tensor-core GEMV over tiles of 16 positions: experts with one partial
    tile, several tiles and a ragged last tile."""
    fam, w, dw = weights("olmoe_decode")
    x = W.make_x(fam, T)
    layer = make_layer(fam, T)
    out, r = run(layer, x, dw, fam.top_k, "tcgemv")
    ref = reference(x, w, fam.top_k)
    check_routing(r, ref, fam.n_experts)
    check_output(out, ref)
    assert T < 300 or ref["counts"].max() > 16  # several tiles per expert


def _check_all_positions(layer, ref, P, H, path):
    """y of every position against the oracle's, expert by expert (every
    tile of every active expert)."""
    y = gpu_y(layer, P, H, path).cpu().numpy().astype(np.float64)
    ref_y = ref["y"].reshape(P, H)[ref["perm"]]
    off = ref["offsets"]
    for e in np.nonzero(ref["counts"])[0]:
        check_expert_y(y[off[e]:off[e + 1]], ref_y[off[e]:off[e + 1]],
                       f"expert {e} ({off[e + 1] - off[e]} positions)")


@pytest.mark.parametrize("T", [1, 16, 64])
def test_wide_decode_tcgemv(T):
    """Every token's output and every position's y (all tiles of all active
    experts, 16-position tiles with ragged tails)."""
    fam, w, dw = weights("wide_decode")
    x = W.make_x(fam, T)
    layer = make_layer(fam, T)
    out, r = run(layer, x, dw, fam.top_k, "tcgemv")
    ref = reference_threaded(x, w, fam.top_k)
    check_routing(r, ref, fam.n_experts)
    check_output(out, ref)
    _check_all_positions(layer, ref, T * fam.top_k, fam.hidden, "tcgemv")


def test_intermediates_match_oracle():
    """Per-kernel parity: h after gate/up + SwiGLU and y after the down GEMV."""
    fam, w, dw = weights("olmoe_decode")
    T, k = 8, fam.top_k
    x = W.make_x(fam, T)
    layer = make_layer(fam, T)
    run(layer, x, dw, k, "gemv")
    ref = reference(x, w, k, keep_h=True)
    P = T * k
    h = layer.debug_buffer("h", torch.float32, (P, fam.inter)).cpu().numpy().astype(np.float64)
    y = layer.debug_buffer("y", torch.float32, (P, fam.hidden)).cpu().numpy().astype(np.float64)
    perm = ref["perm"]
    ref_h = ref["h"].reshape(P, fam.inter)[perm]
    ref_y = ref["y"].reshape(P, fam.hidden)[perm]
    assert np.linalg.norm(h - ref_h) / np.linalg.norm(ref_h) < 1e-4
    assert np.linalg.norm(y - ref_y) / np.linalg.norm(ref_y) < 1e-4


@pytest.mark.parametrize("T,path", [(16, "gemm"), (300, "gemm"), (8, "tcgemv"), (300, "tcgemv")])
def test_tensor_core_paths_y_match_oracle(T, path):
    """Per-kernel parity of the tensor-core paths: y after the down GEMM
    (position order) against the oracle's per-pair y.  Two e4m3 terms hold
    the bf16 x exactly and three keep about 12 bits of h, so y stays near
    1e-5 relative."""
    fam, w, dw = weights("olmoe_decode")
    k = fam.top_k
    x = W.make_x(fam, T)
    layer = make_layer(fam, T)
    out, r = run(layer, x, dw, k, path)
    ref = reference(x, w, k)
    check_routing(r, ref, fam.n_experts)
    check_output(out, ref)
    P = T * k
    if path == "tcgemv":  # one plane per h term; y of a position is their sum
        y3 = layer.debug_buffer("y_terms", torch.float32, (3, P, fam.hidden)).cpu().numpy()
        y = y3.astype(np.float64).sum(axis=0)
    else:
        y = layer.debug_buffer("y", torch.float32, (P, fam.hidden)).cpu().numpy().astype(np.float64)
    ref_y = ref["y"].reshape(P, fam.hidden)[ref["perm"]]
    rel = np.linalg.norm(y - ref_y) / np.linalg.norm(ref_y)
    assert rel < 2e-4, rel


# ------------------------------------------------------------------ full-size workloads

@pytest.mark.parametrize("T", [512, 2048])
def test_olmoe_prefill(T):
    """Every token's output and every position's y: all 128-position tiles of
    all 64 experts, full and ragged."""
    fam, w, dw = weights("olmoe_prefill")
    x = W.make_x(fam, T)
    layer = make_layer(fam, T)
    out, r = run(layer, x, dw, fam.top_k, "auto")
    ref = reference_threaded(x, w, fam.top_k)
    check_routing(r, ref, fam.n_experts)
    check_output(out, ref)
    assert (ref["counts"] > 0).all() and ref["counts"].max() > 2 * ref["counts"].mean()
    _check_all_positions(layer, ref, T * fam.top_k, fam.hidden, layer.resolved_path(T))


@pytest.mark.parametrize("T", [1, 16, 64])
def test_wide_decode(T):
    fam, w, dw = weights("wide_decode")
    x = W.make_x(fam, T)
    layer = make_layer(fam, T)
    out, r = run(layer, x, dw, fam.top_k, "auto")
    ref = reference_threaded(x, w, fam.top_k)
    check_routing(r, ref, fam.n_experts)
    check_output(out, ref)


def test_large_prefill_whole_tiles():
    """Large batch (T = 4096, E = 512, top-12, heavy imbalance): routing of
    every token bit-exact; y of every position of the experts that cover the
    tile classes (the busiest, one with count = 1 mod 128 or nearest, the
    smallest, one in the middle and the last active expert); the output of 64
    tokens spread over the batch and of every token of the busiest expert's
    first 128-position tile."""
    fam, w, dw = weights("large_prefill")
    T, k = 4096, fam.top_k
    x = W.make_x(fam, T)
    layer = make_layer(fam, T)
    out, r = run(layer, x, dw, k, "auto")
    ref_r = reference_threaded(x, w, k, tokens=[])
    check_routing(r, ref_r, fam.n_experts)
    counts, off, perm = ref_r["counts"], ref_r["offsets"], ref_r["perm"]
    assert (counts == 0).any(), "the workload should leave some experts without tokens"
    P, H = T * k, fam.hidden
    experts = tile_class_experts(counts, 128)
    y_ref = oracle_expert_y(x, w, ref_r["idx"], experts)
    y_dev = gpu_y(layer, P, H, layer.resolved_path(T))
    for e in experts:
        rows = y_dev[off[e]:off[e + 1]].cpu().numpy().astype(np.float64)
        check_expert_y(rows, y_ref[e], f"expert {e} ({off[e + 1] - off[e]} positions)")
    del y_dev
    busiest = int(np.argmax(counts))
    tile_tokens = perm[off[busiest]:off[busiest] + 128] // k
    tokens = np.unique(np.concatenate([np.linspace(0, T - 1, 64).astype(np.int64), tile_tokens]))
    assert tokens.size >= 64 + 64
    ref = reference_threaded(x, w, k, tokens=tokens)
    check_output(out, ref, tokens)


@pytest.mark.parametrize("T,path", [(8, "tcgemv"), (8, "gemv"), (2048, "gemm")])
def test_dense_ffn(T, path):
    """A dense (or shared-expert) SwiGLU FFN in the same blockwise-FP8 format
    (dragon.c, "Precision") is the layer with one expert and k = 1: every
    token gets weight 1 and the permutation is the identity.  I = 8192 gives
    64 column blocks of h per tile.  Every token's output and every
    position's y are checked."""
    fam, w, dw = weights("dense_ffn")
    x = W.make_x(fam, T)
    layer = make_layer(fam, T)
    out, r = run(layer, x, dw, 1, path)
    ref = reference_threaded(x, w, 1)
    check_routing(r, ref, 1)
    assert (r["wts"] == 1.0).all() and (r["perm"] == np.arange(T)).all()
    check_output(out, ref)
    _check_all_positions(layer, ref, T, fam.hidden, path)


@pytest.mark.parametrize("T,path", [(300, "gemm"), (8, "tcgemv"), (64, "tcgemv"), (8, "gemv")])
def test_combine_is_the_rank_order_fma_chain(T, path):
    """The combine alone, bit for bit: out equals the host's f32 fma chain in
    rank order over the GPU's own y and routing weights, rounded once to bf16
    (the decode path's y is the f32 sum of its three term planes)."""
    fam, w, dw = weights("olmoe_decode")
    k = fam.top_k
    x = W.make_x(fam, T)
    layer = make_layer(fam, T)
    out, r = run(layer, x, dw, k, path)
    P, H = T * k, fam.hidden
    if path == "tcgemv":
        planes = layer.debug_buffer("y_terms", torch.float32, (3, P, H)).cpu().numpy()
    else:
        planes = layer.debug_buffer("y", torch.float32, (P, H)).cpu().numpy()[None]
    acc = combine_f32(planes, r["inv"], r["wts"])
    want = oracle.round_to_bf16(acc.astype(np.float64))
    assert np.array_equal(out, want), f"{(out != want).sum()} of {out.size} outputs differ"


# ------------------------------------------------------------------ degenerate cases

def _tiny_layer(max_top_k=None, max_tokens=8):
    fam, w, dw = weights("tiny")
    return fam, w, dw, make_layer(fam, max_tokens, max_top_k)


def test_identical_router_rows_tie_to_lower_index():
    fam, w, dw, layer = _tiny_layer()
    rw = w.router_w.copy()
    rw[:] = rw[3]
    w2 = W.LayerWeights(rw, None, w.w13, w.s13, w.w2, w.s2)
    x = W.make_x(fam, 4)
    out, r = run(layer, x, DeviceWeights(w2), fam.top_k)
    assert (r["idx"] == np.arange(fam.top_k)).all()
    assert np.allclose(r["wts"], 1.0 / fam.top_k, rtol=1e-7)
    ref = reference(x, w2, fam.top_k)
    check_routing(r, ref, fam.n_experts)
    check_output(out, ref)


def test_near_ties_are_resolved_exactly():
    """Router rows that differ in one element by one ulp: f32 logits tie or
    flip, the exact order is decided by the f64 recomputation."""
    fam, w, dw, layer = _tiny_layer()
    rw = w.router_w.copy()
    for e in range(1, fam.n_experts):
        rw[e] = rw[0]
        rw[e, e] = np.nextafter(rw[0, e], np.float32(np.inf) if e % 2 else np.float32(-np.inf))
    w2 = W.LayerWeights(rw, None, w.w13, w.s13, w.w2, w.s2)
    x = W.make_x(fam, 4)
    out, r = run(layer, x, DeviceWeights(w2), fam.top_k)
    ref = reference(x, w2, fam.top_k)
    check_routing(r, ref, fam.n_experts)
    check_output(out, ref)


def test_zero_input():
    fam, w, dw, layer = _tiny_layer()
    x = np.zeros((3, fam.hidden), dtype=np.uint16)
    out, r = run(layer, x, dw, fam.top_k)
    assert (out & 0x7FFF == 0).all()
    assert (r["idx"] == np.arange(fam.top_k)).all()


@pytest.mark.parametrize("k", [1, 8])
def test_k_extremes(k):
    fam, w, dw, layer = _tiny_layer(max_top_k=8)
    x = W.make_x(fam, 4)
    out, r = run(layer, x, dw, k)
    ref = reference(x, w, k)
    check_routing(r, ref, fam.n_experts)
    check_output(out, ref)


def test_large_activations_use_exact_power_of_two_scaling():
    fam, w, dw, layer = _tiny_layer()
    x = W.make_x(fam, 4)
    big = (oracle.bf16_to_f64(x) * 2.0 ** 17).astype(np.float32)  # exact in bf16
    xb = (big.view(np.uint32) >> 16).astype(np.uint16)
    assert np.abs(oracle.bf16_to_f64(xb)).max() > 65504
    out, r = run(layer, xb, dw, fam.top_k)
    ref = reference(xb, w, fam.top_k)
    check_routing(r, ref, fam.n_experts)
    check_output(out, ref)


def test_T_equals_max_tokens_and_zero():
    fam, w, dw, layer = _tiny_layer(max_tokens=5)
    x = W.make_x(fam, 5)
    out, r = run(layer, x, dw, fam.top_k)
    check_output(out, reference(x, w, fam.top_k))
    empty = torch.empty((0, fam.hidden), dtype=torch.bfloat16, device="cuda")
    layer.forward(empty, *dw.args(), fam.top_k)
    assert layer.status() == 0


def test_deterministic_bytes():
    fam, w, dw = weights("olmoe_decode")
    x = W.make_x(fam, 8)
    layer = make_layer(fam, 8)
    a = run(layer, x, dw, fam.top_k)
    b = run(layer, x, dw, fam.top_k)
    assert np.array_equal(a[0], b[0])
    for key in a[1]:
        assert np.array_equal(a[1][key], b[1][key])


def test_host_buffer_entry_point_matches():
    fam, w, dw = weights("olmoe_decode")
    T = 8
    x = W.make_x(fam, T)
    layer = make_layer(fam, T)
    out_dev, _ = run(layer, x, dw, fam.top_k)
    xh = torch.from_numpy(x.astype(np.int16)).view(torch.bfloat16).pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    layer.forward_host(xh, *dw.args(), fam.top_k, oh)
    assert np.array_equal(oh.view(torch.int16).numpy().astype(np.uint16), out_dev)


def test_argument_errors():
    fam, w, dw, layer = _tiny_layer(max_tokens=4)
    x = x_dev(W.make_x(fam, 4))
    with pytest.raises(MoEError) as e:
        layer.forward(x, *dw.args(), 3)                  # k > max_top_k
    assert e.value.code == C["MOE_ERR_SHAPE"]
    x5 = x_dev(W.make_x(fam, 5))
    with pytest.raises(MoEError) as e:
        layer.forward(x5, *dw.args(), 2)                 # T > max_tokens
    assert e.value.code == C["MOE_ERR_SHAPE"]
    from fp8_routed_expert_gb300 import lib
    buf = torch.empty(4 * fam.hidden + 8, dtype=torch.bfloat16, device="cuda")
    a = dw.args()
    rc = lib().moe_layer_forward(layer.handle, buf.data_ptr() + 2, 4, a[0].data_ptr(), None,
                                 a[2].data_ptr(), a[3].data_ptr(), a[4].data_ptr(), a[5].data_ptr(),
                                 2, buf.data_ptr(), None)
    assert rc == C["MOE_ERR_ALIGN"]


def test_kernel_timing_api():
    fam, w, dw = weights("olmoe_decode")
    x = W.make_x(fam, 8)
    layer = make_layer(fam, 8)
    layer.set_timing("all")
    n0 = layer.launch_count()
    for _ in range(3):
        run(layer, x, dw, fam.top_k)
    assert layer.resolved_path(8) == "tcgemv"
    # routing logits, selection + sort, fused gate/up + down, combine
    assert layer.launch_count() - n0 == 3 * 4
    for name in ("route", "gate_up", "combine"):
        ms, n = layer.kernel_time(name)
        assert n == 3 and ms > 0, name
    layer.set_timing(["gate_up"])
    run(layer, x, dw, fam.top_k)
    assert layer.kernel_time("gate_up")[1] == 1 and layer.kernel_time("route")[1] == 0
    layer.set_timing(())
