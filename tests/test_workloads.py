"""The seeded input generator (no GPU): determinism, distributions, encoder."""
import numpy as np
import torch

import workloads as W
from workloads import synth


def test_same_data_for_any_thread_count():
    a = W.normal_f32(11, 4, (1000,), 0.02, nthreads=1)
    b = W.normal_f32(11, 4, (1000,), 0.02, nthreads=7)
    assert np.array_equal(a, b)
    c1, s1 = W.blockwise_e4m3(3, 4, 2, 256, 384, 0.02, nthreads=1)
    c2, s2 = W.blockwise_e4m3(3, 4, 2, 256, 384, 0.02, nthreads=5)
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)


def test_streams_are_independent_of_shape():
    # element i of a stream does not depend on how many elements were drawn
    a = W.normal_f32(5, 1, (10,), 1.0)
    b = W.normal_f32(5, 1, (1001,), 1.0)
    assert np.array_equal(a, b[:10])
    assert float(a[3]) == np.float32(synth.lib().gen_normal_at(5, 1, 3))


def test_normal_moments():
    z = W.normal_f32(1, 9, (1 << 20,), 1.0).astype(np.float64)
    assert abs(z.mean()) < 5e-3 and abs(z.std() - 1.0) < 5e-3
    assert abs((z ** 4).mean() - 3.0) < 0.05  # kurtosis of a normal


def test_bf16_activations_are_rounded_normals():
    fam = W.family("tiny")
    x = W.make_x(fam, 4)
    z = W.normal_f32(fam.x_seed(4), 1, (4, fam.hidden), 1.0)
    want = torch.from_numpy(z).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    assert np.array_equal(x, want)


def test_encoder_matches_torch_cast():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(200000) * 50, rng.standard_normal(20000) * 0.01,
                        [448.0, -448.0, 0.0, -0.0, 2.0 ** -10, 3 * 2.0 ** -10, 464.0 - 1e-3]])
    v = np.clip(v, -448, 448).astype(np.float32)
    ours = W.e4m3_encode(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_blockwise_quantisation_contract():
    codes, scales = W.blockwise_e4m3(2, 4, 3, 256, 128, 0.02)
    z = W.normal_f32(2, 4, (3, 256, 128), 0.02)
    for e in range(3):
        for rb in range(2):
            blk = z[e, rb * 128:(rb + 1) * 128]
            s = np.float32(np.abs(blk).max()) / np.float32(448.0)
            assert scales[e, rb, 0] == s
            want = torch.from_numpy(np.clip(blk / s, -448, 448)).to(torch.float8_e4m3fn)
            assert np.array_equal(codes[e, rb * 128:(rb + 1) * 128],
                                  want.view(torch.uint8).numpy())
    assert 0x7F not in codes and 0xFF not in codes


def test_family_shapes():
    for name, fam in W.FAMILIES.items():
        assert fam.hidden % 128 == 0 and fam.inter % 128 == 0
        assert 1 <= fam.top_k <= fam.n_experts
    assert W.parse_workload("olmoe_decode_T8") == (W.family("olmoe_decode"), 8)
