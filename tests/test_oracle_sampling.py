"""Pins of the oracle's sampling step (temperature + top-k with a counter-based generator).

"PersonaPlex native LM audit", section 7 ("One exact generator step"): the generator
samples the text token and each depth position's code; the released defaults are text
temperature 0.7 / top-k 25 and audio temperature 0.8 / top-k 250.  The generator is
Philox4x64-10 (Salmon, Moraes, Dror, Shaw, SC'11), pinned here against NumPy's own,
independently written Philox bit generator; the sampler is pinned by its greedy limits,
its top-k support and the distribution it draws from (counted over many counters).
"""
import math

import numpy as np
import pytest

from oracle import oracle as O


def _numpy_philox_block(counter, key):
    """NumPy's Philox advances its 256-bit counter before each block: start one below."""
    c = sum(int(w) << (64 * i) for i, w in enumerate(counter))
    c = (c - 1) % (1 << 256)
    start = np.array([(c >> (64 * i)) & (2**64 - 1) for i in range(4)], dtype=np.uint64)
    bg = np.random.Philox(key=np.array(key, dtype=np.uint64), counter=start)
    return [int(bg.random_raw()) for _ in range(4)]


def test_philox_matches_numpy_bit_generator():
    rng = np.random.default_rng(7)
    cases = [([0, 0, 0, 0], [0, 0]), ([1, 0, 0, 0], [0, 0]), ([0, 1, 0, 0], [5, 7]),  # borrow across words
             ([2**64 - 1] * 4, [2**64 - 1, 2**64 - 1]), ([12345, 3, 17, 0], [2**63 + 11, 0])]
    for _ in range(20):
        cases.append(([int(v) for v in rng.integers(0, 2**63, 4, dtype=np.uint64)],
                      [int(v) for v in rng.integers(0, 2**63, 2, dtype=np.uint64)]))
    for ctr, key in cases:
        assert O.philox4x64(ctr, key) == _numpy_philox_block(ctr, key), (ctr, key)


def test_uniform_is_top_24_bits_of_first_word():
    for seed, c0, c1, c2 in [(0, 0, 0, 0), (99, 512, 3, 1), (2**64 - 1, 7, 0, 16)]:
        w0 = _numpy_philox_block([c0, c1, c2, 0], [seed, 0])[0]
        u = O.uniform24(seed, c0, c1, c2)
        assert u == (w0 >> 40) / 2.0**24
        assert 0.0 <= u < 1.0


def test_greedy_limits_and_ties():
    lg = np.array([0.5, 2.0, -1.0, 2.0, 1.5])
    for seed in range(5):
        # temperature <= 0 or k <= 1: the argmax, lowest index among equal maxima
        assert O.sample_topk(lg, 0.0, 25, seed, seed, 0, 0)[0] == 1
        assert O.sample_topk(lg, 0.7, 1, seed, seed, 0, 0)[0] == 1
        assert O.sample_topk(lg, -1.0, 250, seed, seed, 0, 0)[0] == 1
    # a tiny temperature concentrates all mass on the maxima; the tie keeps both
    picks = {O.sample_topk(lg, 1e-3, 3, 11, c, 0, 0)[0] for c in range(200)}
    assert picks == {1, 3}


def test_top_k_support_and_cut_ties_to_lower_index():
    lg = np.array([5.0, 1.0, 1.0, 1.0, 4.0])
    seen = set()
    for c in range(2000):
        tok, margin, gap = O.sample_topk(lg, 3.0, 2, 42, c, 0, 0)
        seen.add(tok)
        assert gap == 3.0  # 4th-largest... cut between logit 4.0 (k-th) and 1.0
    assert seen == {0, 4}
    # cut inside a tie: k = 3 keeps index 1 (lowest of the three equal logits), never 2, 3
    seen = {O.sample_topk(lg, 3.0, 3, 42, c, 0, 0)[0] for c in range(4000)}
    assert seen == {0, 1, 4}
    assert O.sample_topk(lg, 3.0, 3, 42, 0, 0, 0)[2] == 0.0


@pytest.mark.parametrize("temperature,top_k", [(0.7, 4), (0.8, 6), (1.0, 8), (2.5, 3)])
def test_distribution_is_softmax_over_top_k_by_counting(temperature, top_k):
    rng = np.random.default_rng(int(temperature * 100) + top_k)
    lg = rng.normal(0.0, 1.5, 8)
    n = 40000
    counts = np.zeros(lg.size)
    for c in range(n):
        counts[O.sample_topk(lg, temperature, top_k, 2024, c, 1, 0)[0]] += 1
    order = sorted(range(lg.size), key=lambda i: (-lg[i], i))
    keep = order[:top_k]
    w = np.array([math.exp((lg[i] - lg[keep[0]]) / temperature) for i in keep])
    p = w / w.sum()
    assert counts[[i for i in range(lg.size) if i not in keep]].sum() == 0
    expected = p * n
    chi2 = float((((counts[keep] - expected) ** 2) / expected).sum())
    # top_k - 1 degrees of freedom; 0.1% tail bound of chi-square with <= 7 dof is < 25
    assert chi2 < 25.0, (chi2, counts[keep], expected)
    # a sampler that ignored the temperature would put this much mass on the top token
    p_t1 = np.exp(lg[keep] - lg[keep[0]])
    p_t1 /= p_t1.sum()
    if abs(temperature - 1.0) > 0.2:
        assert abs(counts[keep[0]] / n - p_t1[0]) > 5 * math.sqrt(p[0] * (1 - p[0]) / n)


def test_inverse_cdf_walks_candidates_in_descending_logit_order():
    # two candidates with weights 3:1 (logit gap T ln 3): u < 3/4 picks the larger
    T = 0.7
    lg = np.array([0.0, T * math.log(3.0)])
    for c in range(300):
        u = O.uniform24(5, c, 0, 0)
        tok, margin, _ = O.sample_topk(lg, T, 2, 5, c, 0, 0)
        assert tok == (1 if u < 0.75 else 0)
        assert abs(margin - abs(u - 0.75)) < 1e-12 or abs(margin - min(u, 1.0 - u)) < 1e-12


def test_depformer_sampling_only_where_not_supplied():
    from full_duplex_speech_moshi_gb300 import inputs as I
    s = I.tiny_shape()
    W = I.make_weights(s, depformer=True)
    specs = I.tensor_specs(s, True)
    orc = O.Oracle(s.asdict(), [W[n] for n, _, _ in specs], depformer=True)
    rng = np.random.default_rng(3)
    h = rng.normal(0, 1, s.D)
    Q = s.dep_steps
    sup = np.array([-1] * 8 + list(rng.integers(0, s.dep_card, Q - 8)), np.int32)
    lg_g, codes_g = orc.depformer_step(h, 5, sup)
    # every position supplied: sampling changes nothing
    lg_a, codes_a, m_a = orc.depformer_step_sampled(h, 5, codes_g.astype(np.int32), 0.8, 250, 9, 3, 0)
    assert np.array_equal(codes_a, codes_g) and np.allclose(lg_a, lg_g) and np.all(np.isinf(m_a))
    # greedy settings reproduce the greedy chain
    lg_b, codes_b, _ = orc.depformer_step_sampled(h, 5, sup, 0.0, 250, 9, 3, 0)
    assert np.array_equal(codes_b, codes_g)
    # sampled: supplied positions keep their codes; each sampled code is the sampler's
    # pick on that position's logits with counter (pos, row, 1 + q)
    lg_c, codes_c, m_c = orc.depformer_step_sampled(h, 5, sup, 0.8, 250, 9, 3, 2)
    assert np.array_equal(codes_c[8:], sup[8:])
    for q in range(8):
        assert codes_c[q] == O.sample_topk(lg_c[q], 0.8, 250, 9, 3, 2, 1 + q)[0]
    assert np.all(np.isfinite(m_c[:8])) and np.all(np.isinf(m_c[8:]))
