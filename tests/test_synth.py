"""The seeded input generator: Philox4x64-10 against numpy's independent implementation of the
same published generator, Box-Muller moments, bf16 rounding, and the workload recipes."""
import numpy as np

import synth


def test_philox_matches_numpy_bit_generator():
    # numpy's Philox advances its 256-bit counter before producing a block, so the block it
    # returns after starting at counter c is Philox(c + 1, key).
    for key in ([1, 2], [0x6D4C6F52, 7], [2**64 - 1, 12345]):
        for start in (0, 5, 2**40):
            bg = np.random.Philox(key=np.array(key, dtype=np.uint64),
                                  counter=np.array([start, 0, 0, 0], dtype=np.uint64))
            ref = bg.random_raw(12).reshape(3, 4)
            for b in range(3):
                got = synth.philox4x64_10([start + 1 + b, 0, 0, 0], key)
                assert np.array_equal(got, ref[b])


def test_raw_words_follow_counter_layout():
    w = synth.raw_u64(11, 22, 40)
    for e in (0, 1, 5, 39):
        assert w[e] == synth.philox4x64_10([e // 4, 0, 0, 0], [11, 22])[e % 4]
    # any sub-range regenerates alone
    assert np.array_equal(synth.raw_u64(11, 22, 9, first=17), w[17:26])


def test_normal_moments_and_subranges():
    z = synth.normal_f64(3, 4, (400_000,))
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    assert abs(((z ** 4).mean()) - 3.0) < 0.05       # normal kurtosis
    assert np.array_equal(synth.normal_f64(3, 4, (100,), first=1234), z[1234:1334])


def test_bf16_rounding_is_nearest_even():
    v = synth.normal_f64(9, 9, (50_000,), std=0.02)
    b = synth.normal_bf16(9, 9, (50_000,), std=0.02)
    f = synth.bf16_bits_to_f32(b).astype(np.float64)
    v32 = v.astype(np.float32).astype(np.float64)
    # nearest: the error is at most half a bf16 ulp of the fp32 value
    ulp = 2.0 ** (np.floor(np.log2(np.abs(v32))) - 7)
    assert np.all(np.abs(f - v32) <= ulp / 2 + 1e-30)


def test_recipes_shapes_and_distributions():
    w = synth.tiny()
    assert w.token_slots.shape == (16, 1) and set(np.unique(w.token_slots)) <= {-1, 0, 1, 2, 3}
    c = synth.compose(T=64)
    for t in range(64):
        row = c.token_slots[t]
        act = row[row >= 0]
        assert len(act) >= 1 and len(set(act.tolist())) == len(act)       # without replacement
        assert np.all(row[len(act):] == -1)                                 # trailing sentinels
    assert np.all((c.scales[c.token_slots >= 0] >= 0.2) & (c.scales[c.token_slots >= 0] <= 1.0))
    plan = synth.mixed_step_plan()
    assert plan["T"] == 4 * 192 + 256
    assert len(plan["slot_of"]) <= 128


def test_admission_rule_defers_new_adapters():
    adm = synth.zipf_admission(300, 1000, 1.1, 5, 123, 9)
    assert len(set(adm)) <= 5 and len(adm) == 300


def test_lm_head_mixture_recipe():
    w = synth.logits(T=200, vocab=512, hidden=256)
    slots, g = w.token_slots, w.scales
    idle = np.all(slots < 0, axis=1)
    assert 0.03 < idle.mean() < 0.2                                       # about 10 % without adapters
    act = ~idle
    assert np.all(slots[act] >= 0) and all(len(set(r)) == w.J for r in slots[act].tolist())
    assert np.allclose(g[act].sum(axis=1), 1.0, atol=1e-6) and np.all(g[act] > 0)   # gate weights
    assert np.all(g[idle] == 0)
    assert {a.rank for a in w.linears[0].adapters.values()} == {8, 16, 32} and w.r_max == 32
    assert w.linears[0].W.shape == (512, 256)
