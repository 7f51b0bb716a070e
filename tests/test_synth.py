"""The shared seeded input generator (no method arithmetic)."""
import numpy as np

import synth


def test_splitmix64_published_vector():
    # splitmix64 seeded with 0: the commonly published first outputs.
    z = synth.splitmix64_stream(0, 4)
    assert [int(x) for x in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
                                   0x06C45D188009454F, 0xF88BB8A8724C81EC]


def test_c_helper_matches_numpy_definition():
    for n in (1, 2, 7, 1000):
        a = synth.normals_f32(99, n)
        b = synth.normals(99, n).astype(np.float32)
        assert np.array_equal(a, b)


def test_normals_moments():
    x = synth.normals_f32(5, 400000).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01


def test_round_bf16_ties_to_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 65504.0],
                    dtype=np.float32)
    out = synth.round_bf16(vals)
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to the even mantissa (1.0)
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: ties to 1 + 2^-6
    assert out.tolist() == [1.0, 1.0, 1.0 + 2 ** -6, 1.0, -2.5, 65536.0]
    assert np.array_equal(out, synth.round_bf16_(vals.copy()))


def test_video_qkv_is_deterministic_and_bf16():
    q1, k1, v1 = synth.video_qkv(1, 2, 3, 4, 5, 64, seed=7)
    q2, k2, v2 = synth.video_qkv(1, 2, 3, 4, 5, 64, seed=7)
    assert np.array_equal(q1, q2) and np.array_equal(k1, k2) and np.array_equal(v1, v2)
    for x in (q1, k1, v1):
        assert np.array_equal(x, synth.round_bf16(x))
    q3, _, _ = synth.video_qkv(1, 2, 3, 4, 5, 64, seed=8)
    assert not np.array_equal(q1, q3)


def test_video_qk_share_modes():
    # q and k of a head share the signal: their correlation is well above 0,
    # while v is independent of both.
    q, k, v = synth.video_qkv(1, 1, 6, 8, 8, 64, seed=3, dtype="f32")
    qq, kk, vv = q.reshape(-1), k.reshape(-1), v.reshape(-1)
    assert np.corrcoef(qq, kk)[0, 1] > 0.5
    assert abs(np.corrcoef(qq, vv)[0, 1]) < 0.05


def test_init_indices_distinct_and_seeded():
    idx = synth.init_indices(2, 3, 500, 64, seed=11)
    assert idx.shape == (2, 3, 64)
    for b in range(2):
        for h in range(3):
            assert len(set(idx[b, h].tolist())) == 64
            assert idx[b, h].min() >= 0 and idx[b, h].max() < 500
    assert np.array_equal(idx, synth.init_indices(2, 3, 500, 64, seed=11))
    full = synth.init_indices(1, 1, 50, 50, seed=1)[0, 0]
    assert sorted(full.tolist()) == list(range(50))
