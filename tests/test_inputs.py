"""The seeded input generator: known-answer stream values, determinism, ranges."""

import numpy as np
import torch

from half_precision_dense_gb300 import inputs


def test_splitmix64_known_answers():
    # The first three outputs of SplitMix64 started from state 0.
    z = inputs.splitmix64(0, 0, 0, 3)
    assert [int(v) for v in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_stream_is_counter_based():
    whole = inputs.splitmix64(5, 1, 0, 1000)
    part = inputs.splitmix64(5, 1, 400, 100)
    assert np.array_equal(whole[400:500], part)
    assert not np.array_equal(inputs.splitmix64(5, 0, 0, 100), inputs.splitmix64(5, 1, 0, 100))
    assert not np.array_equal(inputs.splitmix64(5, 0, 0, 100), inputs.splitmix64(6, 0, 0, 100))


def test_generate_deterministic_and_in_range():
    a = inputs.generate((300, 200), "bf16", 7, 0)
    b = inputs.generate((300, 200), "bf16", 7, 0)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    f = a.float()
    assert f.min() >= -1.0 and f.max() <= 1.0
    assert abs(f.mean().item()) < 0.02
    assert abs(f.var().item() - 1 / 3) < 0.02


def test_uniform_values_are_single_rounded_fp32_draws():
    k = (inputs.splitmix64(3, 1, 0, 5000) >> np.uint64(40)).astype(np.int64)
    f32 = ((k - (1 << 23)) / float(1 << 23)).astype(np.float32)
    want = torch.from_numpy(f32).to(torch.float16)
    got = inputs.generate((50, 100), "f16", 3, 1).reshape(-1)
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_normal_moments():
    g = inputs.generate((512, 512), "bf16", 2, 0, "normal", 1.0).double()
    assert abs(g.mean().item()) < 0.01
    assert abs(g.std().item() - 1.0) < 0.01
    s = inputs.generate((512, 256), "bf16", 3, 1, "normal", 0.02).double()
    assert abs(s.std().item() - 0.02) < 0.001


def test_normal_sub_block_regenerates():
    whole = inputs._normal_f32(9, 0, 0, 101, 1.0)
    part = inputs._normal_f32(9, 0, 33, 51, 1.0)
    assert np.array_equal(whole[33:84], part)


def test_bits_roundtrip():
    a = inputs.generate((17, 9), "f16", 1, 0)
    b = inputs.bits(a)
    assert b.dtype == np.uint16 and b.shape == (17, 9)
    assert torch.equal(inputs.from_bits(b, "f16").view(torch.int16), a.view(torch.int16))


def test_workload_table_shapes():
    w = inputs.WORKLOADS
    assert w["square4096_bf16"][:3] == (4096, 4096, 4096)
    assert w["tails_bf16"][:3] == (1000, 4095, 4104)
    assert w["skinny_bf16"][:3] == (128, 8192, 8192)
    assert w["shortk_bf16"][:3] == (4096, 4096, 64)
    assert w["mlp_up_bf16"][:3] == (16384, 14336, 4096)
    assert w["mlp_down_bf16"][:3] == (16384, 4096, 14336)
