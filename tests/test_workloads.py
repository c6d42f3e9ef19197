"""The benchmark workloads and their seeded inputs: the algorithmic bytes and flops the roofline
divides by, against the figures stated for each shape (A bf16 read + B e2m1 and e8m0 read + C bf16
write; 2MNK), and the input recipe (normal A and B, B scaled to sigma 0.02 on the 64x7168x2048
shape, 5 % of A's 1x32 blocks x1e3 and another 5 % zeroed on the 32x4096x512 shape)."""
import pytest
import torch

from block_scaled_mxfp4_bf16_gb300 import workloads

STATED = {   # name: (algorithmic bytes, 2MNK)
    "M16_N3072_K1536": (2_654_208, 1.510e8),
    "M8_N2112_K7168": (8_190_976, 2.422e8),
    "M32_N4096_K512": (1_409_024, 1.342e8),
    "M64_N7168_K2048": (8_978_432, 1.879e9),
    "M256_N4096_K7168": (21_364_736, 1.503e10),
}


@pytest.mark.parametrize("name", list(STATED))
def test_roofline_units_match_the_stated_figures(name):
    w = workloads.by_name(name)
    nbytes, flops = STATED[name]
    assert w.algorithmic_bytes == nbytes
    assert abs(w.flops - flops) / flops < 1e-3


def test_inputs_are_seeded_and_deterministic():
    w = workloads.by_name("M16_N3072_K1536")
    a1, b1 = workloads.make_inputs(w, seed=0)
    a2, b2 = workloads.make_inputs(w, seed=0)
    assert a1.dtype == b1.dtype == torch.bfloat16
    assert tuple(a1.shape) == (16, 1536) and tuple(b1.shape) == (3072, 1536)
    assert torch.equal(a1, a2) and torch.equal(b1, b2)
    a3, _ = workloads.make_inputs(w, seed=1)
    assert not torch.equal(a1, a3)


def test_outlier_and_zero_blocks_of_the_short_k_shape():
    w = workloads.by_name("M32_N4096_K512")
    a, _ = workloads.make_inputs(w, seed=0)
    amax = a.float().abs().reshape(-1, 32).amax(dim=1)     # 512 blocks of 1x32
    n5 = 512 * 5 // 100
    assert int((amax == 0).sum()) == n5                    # zeroed blocks
    assert int((amax > 100).sum()) == n5                   # x1e3 blocks (N(0,1) blocks stay below 100)


def test_weight_scale_of_the_wide_shape():
    w = workloads.by_name("M64_N7168_K2048")
    a, b = workloads.make_inputs(w, seed=0)
    assert abs(float(b.float().std()) - 0.02) < 0.001
    assert abs(float(a.float().std()) - 1.0) < 0.02


def test_workloads_named_by_shape():
    # any M<m>_N<n>_K<k> names a plain workload of that shape (sigma 1, no outliers); listed
    # names keep their own recipes; anything else is unknown
    w = workloads.by_name("M2048_N4096_K7168")
    assert (w.M, w.N, w.K, w.b_sigma, w.outlier_blocks) == (2048, 4096, 7168, 1.0, False)
    assert workloads.by_name("M64_N7168_K2048").b_sigma == 0.02
    for bad in ("M0_N128_K256", "M8_N2112", "foo", "M8_N2112_K7168x"):
        with pytest.raises(KeyError):
            workloads.by_name(bad)
