"""The synthetic inputs follow their stated recipe (CPU, small sizes).

Checks the seeded generator against the workload descriptions: weights N(mean, std) rounded to
BF16, changes at Bernoulli(rate) positions, the 97 / 2.9 / 0.1 mantissa / exponent / sign mix,
row clustering, the MoE hot-expert share, the dense additive rule, and determinism.  The
class of each change is read from the bit fields directly (no codec code involved).
"""
import math

import torch

import workloads as W


def _bits(t):
    return t.reshape(-1).view(torch.int16).to(torch.int32) & 0xFFFF


def test_pair_is_deterministic_and_seeded_per_tensor():
    s = W.Spec("t", (257, 129), tid=3)
    a1, b1 = W.make_pair(s, device="cpu")
    a2, b2 = W.make_pair(s, device="cpu")
    assert torch.equal(_bits(a1), _bits(a2)) and torch.equal(_bits(b1), _bits(b2))
    a3, _ = W.make_pair(W.Spec("t", (257, 129), tid=4), device="cpu")
    assert not torch.equal(_bits(a1), _bits(a3))


def test_rate_and_mutation_mix():
    n = 1 << 22
    s = W.Spec("t", (n,), rate=0.02, tid=11)
    old, new = W.make_pair(s, device="cpu")
    x = _bits(old) ^ _bits(new)
    changed = int((x != 0).sum())
    # Bernoulli(0.02) over n positions (exponent steps are skipped only at fields 0 and 255,
    # which N(0, 0.02) weights do not reach)
    mean, sd = 0.02 * n, math.sqrt(0.02 * 0.98 * n)
    assert abs(changed - mean) < 6 * sd
    mant = int(((x != 0) & ((x & 0xFF80) == 0)).sum())
    sign = int((x == 0x8000).sum())
    expo = changed - mant - sign
    assert abs(mant / changed - 0.97) < 0.005
    assert abs(expo / changed - 0.029) < 0.003
    assert abs(sign / changed - 0.001) < 0.0008
    # exponent changes move the field by exactly one and touch nothing else
    e_old, e_new = (_bits(old) >> 7) & 0xFF, (_bits(new) >> 7) & 0xFF
    em = ((x & 0x7F80) != 0) & ((x & 0x807F) == 0)
    assert int(em.sum()) == expo
    assert bool(((e_old[em] - e_new[em]).abs() == 1).all())


def test_weight_distribution_and_norm_init():
    old, _ = W.make_pair(W.Spec("w", (1 << 20,), tid=5), device="cpu")
    f = old.float()
    assert abs(float(f.mean())) < 1e-4 and abs(float(f.std()) - 0.02) < 2e-4
    norm, _ = W.make_pair(W.Spec("n", (4096,), std=1e-3, mean=1.0, tid=6), device="cpu")
    g = norm.float()
    assert abs(float(g.mean()) - 1.0) < 1e-4 and float(g.std()) < 2e-3


def test_clustered_changes_stay_in_hot_rows():
    s = W.Spec("c", (1000, 256), rate=0.2, rows_hot=0.1, tid=7)
    old, new = W.make_pair(s, device="cpu")
    rows = ((_bits(old) ^ _bits(new)) != 0).reshape(1000, 256).any(1)
    assert int(rows.sum()) <= 100 and int(rows.sum()) >= 95


def test_additive_rule_in_bf16_arithmetic():
    # new = old + 1e-3 * N(0, 1) in BF16 arithmetic, as in the pages' API snippet: a BF16 ulp near
    # |x| = 1 is 2^-7, so most 1e-3 steps round away and about 22% of the elements change; those
    # that do change their mantissa, and some (steps across a power of two) their exponent
    s = W.Spec("d", (1 << 20,), kind="additive", tid=0)
    old, new = W.make_pair(s, device="cpu")
    x = _bits(old) ^ _bits(new)
    frac = float((x != 0).float().mean())
    assert 0.18 < frac < 0.28
    rare = int(((x & 0xFF80) != 0).sum()) / int((x != 0).sum())
    assert 0.01 < rare < 0.1
    d = (new.float() - old.float()).abs()
    assert float(old.float().std()) > 0.99 and float(d.max()) <= 2 ** -6


def test_workload_shapes():
    d = W.dense7b()
    assert len(d) == 1 + 32 * 9 + 2 and sum(s.numel for s in d) == 6_738_415_616
    m = W.moe30b()
    assert len(m) == 1 + 48 * (128 * 3 + 5) + 1
    hot = [s for s in m if s.rate == max(x.rate for x in m)]
    n_tot = sum(s.numel for s in m)
    changed = sum(s.rate * s.numel for s in m)
    assert abs(changed / n_tot - 0.03) < 1e-9
    assert abs(sum(s.rate * s.numel for s in hot) / changed - 0.8) < 1e-9
    assert len(hot) == 48 * 8 * 3
    sw = W.sweep14336()
    assert [s.rate for s in sw[:5]] == list(W.SWEEP_RATES) and sw[5].rows_hot == 0.1
    assert W.single_1m()[0].numel == 1 << 20 and W.dense1g()[0].numel == 1 << 29
