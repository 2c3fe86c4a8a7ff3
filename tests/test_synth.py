"""The seeded input generators (synth/): the random streams against their published definitions,
the bf16 rounding against PyTorch's, and the input recipe (shapes, distributions, document
layouts) that the tests, the benchmark and the oracle all draw from."""
import math

import numpy as np
import pytest

import synth

MASK = (1 << 64) - 1


def _splitmix64_scalar(state, n):
    """splitmix64 from its published definition (Steele, Lea and Flood 2014): add the golden
    gamma to the state, then the two xor-shift-multiply rounds and a final xor-shift."""
    out = []
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & MASK
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
        out.append(z ^ (z >> 31))
    return out


def test_splitmix64_known_answer_and_vectorised_stream():
    # the generator's published first outputs from state 0
    assert _splitmix64_scalar(0, 4) == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F,
                                        0xF88BB8A8724C81EC]
    for seed, stream in [(1001, 1), (1005, 8), (7, 100)]:
        key = int(synth._mix_seed(seed, stream))
        got = [int(x) for x in synth.splitmix64(seed, stream, 64)]
        assert got == _splitmix64_scalar(key, 64)
    # streams and seeds are distinct sequences
    a = synth.splitmix64(1001, 1, 1000)
    assert not np.array_equal(a, synth.splitmix64(1001, 2, 1000))
    assert not np.array_equal(a, synth.splitmix64(1002, 1, 1000))


def test_uniform_and_normal_draws():
    n = 1 << 18
    u = synth.uniform01(1234, 3, n)
    assert u.min() > 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 5 * math.sqrt(1 / 12 / n)
    x = synth.normal(1234, 4, n)
    assert abs(x.mean()) < 5 / math.sqrt(n)
    assert abs(x.var() - 1.0) < 5 * math.sqrt(2 / n)
    # the two members of each Box-Muller pair are uncorrelated
    assert abs(np.corrcoef(x[0::2], x[1::2])[0, 1]) < 5 / math.sqrt(n / 2)
    # fourth moment of a standard normal is 3
    assert abs((x ** 4).mean() - 3.0) < 5 * math.sqrt(96 / n)
    # odd lengths and reproducibility
    np.testing.assert_array_equal(synth.normal(9, 1, 7), synth.normal(9, 1, 8)[:7])


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-30, 30, 100000))).astype(np.float32)
    # exact ties (lower 16 bits 0x8000) with even and odd kept parts, both signs, and signed zeros
    hi = (np.uint32(0x3F80) | rng.integers(0, 128, 2000, dtype=np.uint32)) << np.uint32(16)
    ties = hi | np.uint32(0x8000)
    x = np.concatenate([x, ties.view(np.float32), (ties | np.uint32(0x80000000)).view(np.float32),
                        np.float32([0.0, -0.0, 1.0, -2.5])])
    ours = synth.to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    # the round trip is exact for values that are already bf16
    back = synth.bf16_bits_to_f32(ours)
    np.testing.assert_array_equal(synth.to_bf16_bits(back), ours)


def test_problem_recipe():
    T, Hk, Hv = 4096, 2, 8
    p = synth.make_problem("recipe", 2024, [1000, 0, 3096], Hk, Hv, n_init=2, init_idx=[-1, 0, 1],
                           with_dout=True, with_dfinal=True)
    assert p.T == T and p.N == 3 and list(p.cu_seqlens) == [0, 1000, 1000, 4096]
    assert p.q.shape == p.k.shape == (T, Hk, 128) and p.v.shape == p.dout.shape == (T, Hv, 128)
    assert p.g.shape == p.beta.shape == (T, Hv) and p.g.dtype == np.float32 and p.beta.dtype == np.float32
    assert p.initial_state.shape == (2, Hv, 128, 128) and p.dfinal.shape == (3, Hv, 128, 128)
    f = p.as_f64()
    # q, k: unit rows per (token, head) before one bf16 rounding, q scaled by 1/sqrt(128)
    nq = np.linalg.norm(f["q"], axis=-1) * math.sqrt(128)
    nk = np.linalg.norm(f["k"], axis=-1)
    assert np.abs(nq - 1).max() < 4e-3 and np.abs(nk - 1).max() < 4e-3
    # v and dO: standard normal, rounded to bf16
    for x in (f["v"], f["dout"]):
        assert abs(x.mean()) < 0.01 and abs(x.var() - 1) < 0.01
    # g = log sigmoid(u), u ~ N(2, 1): negative, with the mean of the exact expectation
    uu = np.linspace(-10, 14, 200001)
    dens = np.exp(-0.5 * (uu - 2.0) ** 2) / math.sqrt(2 * math.pi)
    eg = np.trapezoid(-np.logaddexp(0.0, -uu) * dens, uu)
    assert (p.g < 0).all()
    assert abs(f["g"].mean() - eg) < 5 * f["g"].std() / math.sqrt(T * Hv)
    # beta = sigmoid(w), w ~ N(0, 1): in (0, 1), symmetric about 1/2
    assert (p.beta > 0).all() and (p.beta < 1).all()
    assert abs(f["beta"].mean() - 0.5) < 5 * f["beta"].std() / math.sqrt(T * Hv)
    # pool states N(0, 1) x 0.1
    assert abs(p.initial_state.std() - 0.1) < 0.002
    # a seed gives the same bits; another seed other bits
    p2 = synth.make_problem("recipe", 2024, [1000, 0, 3096], Hk, Hv, n_init=2, with_dout=True, with_dfinal=True)
    for a in ("q", "k", "v", "g", "beta", "dout", "initial_state", "dfinal"):
        np.testing.assert_array_equal(getattr(p, a), getattr(p2, a))
    p3 = synth.make_problem("recipe", 2025, [1000, 0, 3096], Hk, Hv)
    assert not np.array_equal(p.q, p3.q) and not np.array_equal(p.g, p3.g)


def test_gqa_ratio_must_divide():
    with pytest.raises(ValueError):
        synth.make_problem("bad", 1, [10], 3, 4)


@pytest.mark.parametrize("total,n", [(16384, 12), (1024, 12), (48000, 12)])
def test_lognormal_lengths_fill_the_buffer(total, n):
    lens = synth.lognormal_lengths(1002, n, total)
    assert len(lens) == n and sum(lens) == total
    assert min(lens) >= 64 and max(lens) <= 4096
    assert lens == synth.lognormal_lengths(1002, n, total)
    with pytest.raises(ValueError):
        synth.lognormal_lengths(1002, n, n * 4096 + 1)


def test_uniform_int_lengths_cover_the_range():
    lens = synth.uniform_int_lengths(77, 40000, 2, 5)
    assert min(lens) == 2 and max(lens) == 5
    counts = np.bincount(lens)[2:]
    assert np.abs(counts - 10000).max() < 5 * math.sqrt(40000 * 0.25 * 0.75)
    big = synth.uniform_int_lengths(1004, 16, 2048, 6144)
    assert all(2048 <= x <= 6144 for x in big)


def test_workload_layouts_at_small_sizes():
    s = synth.workload_single(T=300, Hk=1, Hv=2)
    assert s.N == 1 and s.T == 300 and s.init_idx is None and s.initial_state is None
    pk = synth.workload_packed(total=2048, n_docs=12, Hk=1, Hv=2)
    assert pk.N == 12 and pk.T == 2048 and np.all(np.diff(pk.cu_seqlens) >= 64)
    lg = synth.workload_long(T=640, Hk=1, Hv=2)
    assert lg.N == 1 and lg.T == 640
    fk = synth.workload_fork(prefix=128, n_branch=3, lo=64, hi=96, Hk=1, Hv=2)
    lens = np.diff(fk.cu_seqlens)
    assert lens[0] == 128 and all(64 <= x <= 96 for x in lens[1:])
    assert list(fk.init_idx) == [-1, 0, 0, 0] and fk.n_init == 0  # every branch forks document 0
    tr = synth.workload_train(n_docs=2, doc_len=100, Hk=1, Hv=2)
    assert list(tr.cu_seqlens) == [0, 100, 200] and tr.dout is not None and tr.dout.shape == (200, 2, 128)


def test_f16_rounding_matches_torch():
    torch = __import__("pytest").importorskip("torch")
    import numpy as np
    x = np.random.default_rng(5).standard_normal(4096) * np.exp(np.random.default_rng(6).uniform(-12, 10, 4096))
    ours = synth.to_f16_bits(x)
    ref = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = synth.f16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.float16).float().numpy())
