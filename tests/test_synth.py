"""The seeded generator: its tensor form equals its scalar definition, slices equal the whole,
and the draws have the stated distributions."""
import numpy as np
import torch

import synth


def test_word_matches_scalar_definition():
    k0, k1 = synth.key(1234, synth.TAG_W13)
    cs = [0, 1, 2, 12345, (1 << 32) - 1, 1 << 32, (1 << 33) + 77, 7_516_192_767]
    got = synth.word(torch.tensor(cs, dtype=torch.int64), k0, k1).tolist()
    assert got == [synth.word_int(c, k0, k1) for c in cs]
    assert all(0 <= g < (1 << 32) for g in got)


def test_normal_draws_are_standard_normal():
    """Moments, tails and the distribution function of N(0, 1): a bounded bell (such as a sum of
    a few uniforms) fails the tail and kurtosis checks, a wrong branch or scale the moments."""
    from scipy.special import ndtr
    n = 1 << 20
    x = synth.normal_f32(5, synth.TAG_X, (n,), 1.0).double().numpy()
    assert abs(x.mean()) < 0.005
    assert abs(x.std() - 1.0) < 0.005
    kurt = np.mean((x - x.mean()) ** 4) / x.var() ** 2
    assert abs(kurt - 3.0) < 0.05
    # P(|z| > 3) = 0.0026998, P(|z| > 4) = 6.33e-5: about 2831 +- 53 and 66 +- 8 of 2**20
    assert 2550 <= int((np.abs(x) > 3).sum()) <= 3110
    assert 30 <= int((np.abs(x) > 4).sum()) <= 110
    # 32-bit uniforms bound the draws at sqrt(2 * 32 ln 2)
    assert np.abs(x).max() <= (64 * np.log(2)) ** 0.5 + 1e-6
    # Kolmogorov-Smirnov distance to the normal CDF (the 1 % critical value is 1.63 / sqrt(n))
    xs = np.sort(x)
    cdf = ndtr(xs)
    i = np.arange(1, n + 1)
    ks = max(np.max(i / n - cdf), np.max(cdf - (i - 1) / n))
    assert ks < 1.63 / n ** 0.5
    # a known draw from the definition: z for element 0 of this stream
    k0, k1 = synth.key(5, synth.TAG_X)
    u1 = (synth.word_int(0, k0, k1) + 1) / 2.0 ** 32
    u2 = synth.word_int(1, k0, k1) / 2.0 ** 32
    import math
    z0 = math.sqrt(-2.0 * math.log(u1)) * math.cos(2.0 * math.pi * u2)
    assert abs(x[0] - z0) <= 2.0 ** -23 * max(1.0, abs(z0))
    w = synth.normal_bf16(5, synth.TAG_W2, (1 << 18,), 0.02).float()
    assert abs(w.std().item() - 0.02) < 0.0002


def test_uniform_range():
    b = synth.uniform_sym_f32(0, synth.TAG_BIAS, 100000, 0.1)
    assert b.min().item() >= -0.1 and b.max().item() < 0.1
    assert abs(b.mean().item()) < 0.002


def test_slices_equal_whole_tensor():
    cfg = synth.MoEConfig("t", T=8, d=256, E=3, k=1, n_group=1, topk_group=1, d_ff=128,
                          d_ff_shared=0, R=1, route_scale=1.0, seed=9)
    W = synth.make_expert_weights(cfg)
    for e in range(3):
        s = synth.expert_weight_slice(cfg, e)
        assert torch.equal(s["w13"], W["w13"][e]) and torch.equal(s["w2"], W["w2"][e])
    cfg8 = synth.MoEConfig("t", T=8, d=256, E=3, k=1, n_group=1, topk_group=1, d_ff=128,
                           d_ff_shared=128, R=1, route_scale=1.0, act="fp8", w="fp8", seed=9)
    W8 = synth.make_expert_weights(cfg8)
    s = synth.expert_weight_slice(cfg8, 2)
    assert torch.equal(s["w13"], W8["w13"][2]) and torch.equal(s["w13_s"], W8["w13_s"][2])
    assert W8["ws13"].shape == (256, 256) and W8["ws2_s"].shape == (2, 1)


def test_fp8_block_weights_dequantise_close_to_draws():
    q, s = synth.fp8_block_weights(3, synth.TAG_W13, 1, 256, 256, 0.02)
    w = synth.normal_f32(3, synth.TAG_W13, (256, 256), 0.02)
    deq = q[0].view(torch.float8_e4m3fn).float() * s[0].repeat_interleave(128, 0).repeat_interleave(128, 1)
    assert (deq - w).abs().max().item() <= 0.07 * w.abs().max().item()
    # each block's largest magnitude maps to the largest code
    blk = q[0].view(torch.float8_e4m3fn).float().abs().view(2, 128, 2, 128).amax(dim=(1, 3))
    assert torch.all(blk == 448.0)


def test_permutation_and_zipf_bias():
    p = synth.permutation(1, synth.TAG_PERM, 256)
    assert sorted(p.tolist()) == list(range(256))
    cfg = synth.CONFIGS["dsv3_skew_prefill"]
    b = synth.zipf_bias(cfg).numpy()
    assert abs(float(b.mean())) < 1e-5
    assert int(np.argmax(b)) == int(synth.permutation(cfg.seed, synth.TAG_PERM, cfg.E)[0])


def test_configs_follow_the_stated_workloads():
    c = synth.CONFIGS
    assert (c["tiny"].T, c["tiny"].d, c["tiny"].E, c["tiny"].k, c["tiny"].R) == (16, 256, 16, 2, 2)
    d = c["dsv3_decode"]
    assert (d.T, d.d, d.E, d.k, d.n_group, d.topk_group, d.d_ff, d.d_ff_shared, d.R) == \
        (64, 7168, 256, 8, 8, 4, 2048, 2048, 8)
    assert d.route_scale == 2.5 and d.cap == 64
    assert synth.SWEEP_T == [8, 16, 32, 64, 128, 256, 512, 1024]
    assert c["dsv3_skew_prefill"].T == 4096 and c["dsv3_fp8_prefill"].T == 16384
