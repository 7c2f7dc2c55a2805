"""Pins for the fp64 oracle: each check ties it to something the pages or plain mathematics fix,
never to itself. A mutation test compiles altered copies of the oracle source and shows that
these pins catch the plausible mistakes (wrong factor, dropped term, transposed index...)."""
import os
import shutil
import subprocess
import tempfile
from types import SimpleNamespace

import numpy as np
import pytest

import oracle
from oracle import memory
from tests.conftest import read_golden


# ----------------------------------------------------------------------------- helpers
def _hand_case(path="hand_two_slot_rslora.txt"):
    g = read_golden(path)
    d = {}
    slots = {}
    cur = None
    for key, vals in g:
        if key == "slot":
            cur = int(vals[0])
            kv = dict(zip(vals[1::2], vals[2::2]))
            slots[cur] = SimpleNamespace(rank=int(kv["rank"]), alpha=float(kv["alpha"]),
                                         rslora=bool(int(kv["rslora"])))
        else:
            d[key] = vals
    T, K, D, J, S = (int(d[k][0]) for k in ("T", "K", "D", "J", "n_slots"))
    f = lambda k: np.array([float(v) for v in d[k]])  # noqa: E731
    for s, ad in slots.items():
        ad.A = f(f"A{s}").reshape(ad.rank, K)
        ad.B = f(f"B{s}").reshape(D, ad.rank)
    return dict(T=T, K=K, D=D, J=J, S=S, x=f("x").reshape(T, K), W=f("W").reshape(D, K),
                slots=np.array([int(v) for v in d["token_slots"]]).reshape(T, J),
                scales=f("scales").reshape(T, J), adapters=slots,
                y=f("y").reshape(T, D), y_plain=f("y_plain").reshape(T, D))


def _random_case(seed, T=7, K=24, D=20, J=2, S=4, ranks=(3, 5, 2, 4)):
    rng = np.random.default_rng(seed)
    ads = {s: SimpleNamespace(A=rng.standard_normal((ranks[s], K)), B=rng.standard_normal((D, ranks[s])),
                              rank=ranks[s], alpha=float(rng.integers(1, 9)), rslora=bool(s % 2))
           for s in range(S)}
    slots = rng.integers(-1, S, size=(T, J))
    scales = rng.uniform(0.2, 1.0, size=(T, J))
    return dict(x=rng.standard_normal((T, K)), W=rng.standard_normal((D, K)), slots=slots,
                scales=scales, adapters=ads, S=S, T=T, K=K, D=D, J=J)


def _factor(ad):
    return ad.alpha / (np.sqrt(ad.rank) if ad.rslora else ad.rank)


# ----------------------------------------------------------------------------- hand example
def test_hand_example_two_slots_with_rslora_and_sentinel():
    c = _hand_case()
    y = oracle.linear(c["x"], c["W"], c["slots"], c["adapters"], c["S"], scales=c["scales"])
    assert np.array_equal(y, c["y"])          # every intermediate is exact in binary


def test_hand_example_plain_lora_factor():
    c = _hand_case()
    c["adapters"][1].rslora = False
    y = oracle.linear(c["x"], c["W"], c["slots"], c["adapters"], c["S"], scales=c["scales"])
    assert np.array_equal(y, c["y_plain"])


def test_hand_example_row_and_column_selection():
    c = _hand_case()
    y = oracle.linear(c["x"], c["W"], c["slots"], c["adapters"], c["S"], scales=c["scales"],
                      rows=[2, 0], cols=[1])
    assert np.array_equal(y, c["y"][[2, 0]][:, [1]])


# ----------------------------------------------------------------------------- invariants
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_sentinel_and_zero_scale_rows_equal_base_exactly(seed):
    c = _random_case(seed)
    slots, scales = c["slots"].copy(), c["scales"].copy()
    slots[0, :] = -1                      # sentinel row
    scales[1, :] = 0.0                    # zero-scale row
    y = oracle.linear(c["x"], c["W"], slots, c["adapters"], c["S"], scales=scales)
    base = oracle.linear(c["x"], c["W"], np.full_like(slots, -1), {}, c["S"])
    assert np.array_equal(y[0], base[0])
    assert np.array_equal(y[1], base[1])
    assert np.array_equal(base, c["x"] @ c["W"].T) or np.allclose(base, c["x"] @ c["W"].T, rtol=1e-13)


@pytest.mark.parametrize("seed", [3, 4])
def test_merge_identity(seed):
    # "Multi-LoRA Serving Explained": W x + s B(A x) == (W + s B A) x (the page's check prints
    # a maximum difference of about 4.3e-14 on a 512 x 512 layer).
    c = _random_case(seed, J=1)
    ad = c["adapters"][1]
    slots = np.full((c["T"], 1), 1)
    y = oracle.linear(c["x"], c["W"], slots, c["adapters"], c["S"])
    W_merged = c["W"] + _factor(ad) * (ad.B @ ad.A)
    y_merged = c["x"] @ W_merged.T
    assert np.max(np.abs(y - y_merged)) <= 1e-12 * np.max(np.abs(y_merged))


@pytest.mark.parametrize("seed", [5, 6])
def test_two_adapters_equal_their_cat_merge(seed):
    # RFC 51940, Testing: composition with fixed scales is identical to PEFT's rank-concatenated
    # ("cat") merge; here A_cat = [A_a; A_b], B_cat = [c_a B_a | c_b B_b], factor 1.
    c = _random_case(seed, J=2)
    a, b = c["adapters"][0], c["adapters"][3]
    s_a, s_b = 0.7, 0.4
    slots = np.tile([0, 3], (c["T"], 1))
    scales = np.tile([s_a, s_b], (c["T"], 1))
    y = oracle.linear(c["x"], c["W"], slots, c["adapters"], c["S"], scales=scales)
    cat = SimpleNamespace(A=np.vstack([a.A, b.A]),
                          B=np.hstack([s_a * _factor(a) * a.B, s_b * _factor(b) * b.B]),
                          rank=a.rank + b.rank, alpha=float(a.rank + b.rank), rslora=False)
    y_cat = oracle.linear(c["x"], c["W"], np.zeros((c["T"], 1)), {0: cat}, 1)
    assert np.max(np.abs(y - y_cat)) <= 1e-12 * np.max(np.abs(y_cat))


@pytest.mark.parametrize("rslora", [False, True])
def test_sliced_adapter_equals_its_block_diagonal_form(rslora):
    # A fused linear with one adapter per output slice equals one adapter of rank n r with
    # A = [A_1; ...; A_n] and block-diagonal B (slice i's rows hold B_i in columns i r ..), whose
    # factor is that of the slices (alpha scaled so that alpha' / (n r) or alpha' / sqrt(n r)
    # equals alpha / r or alpha / sqrt(r)). Also: each slice's outputs differ from the base only
    # through that slice's own adapter.
    rng = np.random.default_rng(31)
    T, K, J, S, r = 6, 20, 2, 3, 3
    widths = [7, 4, 5]
    D = sum(widths)
    x, W = rng.standard_normal((T, K)), rng.standard_normal((D, K))
    sliced = {}
    for s in range(S):
        alpha = float(rng.integers(1, 9))
        sliced[s] = [SimpleNamespace(A=rng.standard_normal((r, K)), B=rng.standard_normal((w, r)), rank=r,
                                     alpha=alpha, rslora=rslora) for w in widths]
    slots = rng.integers(-1, S, size=(T, J))
    scales = rng.uniform(0.2, 1.0, size=(T, J))
    y = oracle.linear_sliced(x, W, slots, sliced, S, widths, scales=scales)
    n = len(widths)
    whole = {}
    for s, parts in sliced.items():
        B = np.zeros((D, n * r))
        off = 0
        for i, (w, p) in enumerate(zip(widths, parts)):
            B[off:off + w, i * r:(i + 1) * r] = p.B
            off += w
        a0 = parts[0].alpha
        whole[s] = SimpleNamespace(A=np.vstack([p.A for p in parts]), B=B, rank=n * r,
                                   alpha=a0 * (np.sqrt(n) if rslora else n), rslora=rslora)
    y_whole = oracle.linear(x, W, slots, whole, S, scales=scales)
    assert np.max(np.abs(y - y_whole)) <= 1e-12 * np.max(np.abs(y_whole))
    # slice 1 alone: its adapter, written out
    t, (s0, s1) = 2, slots[2]
    lo, hi = widths[0], widths[0] + widths[1]
    ref = W[lo:hi] @ x[t]
    for j, s in enumerate((s0, s1)):
        if s >= 0:
            p = sliced[s][1]
            ref = ref + scales[t, j] * _factor(p) * (p.B @ (p.A @ x[t]))
    assert np.max(np.abs(y[t, lo:hi] - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_output_is_linear_in_the_scale():
    c = _random_case(7, J=1)
    slots = np.full((c["T"], 1), 2)
    ys = {s: oracle.linear(c["x"], c["W"], slots, c["adapters"], c["S"], scales=np.full((c["T"], 1), s))
          for s in (0.0, 1.0, 0.37)}
    lhs, rhs = ys[0.37] - ys[0.0], 0.37 * (ys[1.0] - ys[0.0])
    assert np.max(np.abs(lhs - rhs)) <= 1e-12 * np.max(np.abs(ys[1.0]))


def test_zero_padding_to_max_rank_changes_nothing():
    # "Multi-LoRA Serving Explained", max-lora-rank section: a small adapter copied into the
    # top-left corner of a zero slot gives the same output (the page prints True). The factor
    # is kept at the adapter's own alpha / r (the padding does not change the rank).
    c = _random_case(8, J=1)
    ad = c["adapters"][2]
    R = 9
    pad = SimpleNamespace(A=np.zeros((R, c["K"])), B=np.zeros((c["D"], R)), rank=R,
                          alpha=_factor(ad) * R, rslora=False)
    pad.A[:ad.rank] = ad.A
    pad.B[:, :ad.rank] = ad.B
    slots = np.full((c["T"], 1), 0)
    y = oracle.linear(c["x"], c["W"], slots, {0: ad}, 1)
    y_pad = oracle.linear(c["x"], c["W"], slots, {0: pad}, 1)
    assert np.max(np.abs(y - y_pad)) <= 1e-12 * np.max(np.abs(y))


def test_duplicate_slot_in_one_token_counts_twice():
    c = _random_case(9, J=2)
    once = oracle.linear(c["x"], c["W"], np.tile([1, -1], (c["T"], 1)), c["adapters"], c["S"])
    twice = oracle.linear(c["x"], c["W"], np.tile([1, 1], (c["T"], 1)), c["adapters"], c["S"])
    base = oracle.linear(c["x"], c["W"], np.full((c["T"], 2), -1), {}, c["S"])
    assert np.allclose(twice - base, 2 * (once - base), rtol=1e-12, atol=1e-12)


def test_batched_result_equals_per_request_merged_result():
    # The page's six-token demo: gathering each token's adapter in one batch equals running
    # each request alone with its merged weight (and the -1 token with the base weight).
    rng = np.random.default_rng(1)
    d, R = 32, 6
    ranks = (4, 6, 2, 6)
    ads = {s: SimpleNamespace(A=rng.standard_normal((r, d)) * 0.05, B=rng.standard_normal((d, r)) * 0.05,
                              rank=r, alpha=float(r), rslora=False) for s, r in enumerate(ranks)}
    ids = np.array([2, 0, -1, 2, 3, 0])
    X = rng.standard_normal((6, d))
    W = rng.standard_normal((d, d))
    y = oracle.linear(X, W, ids.reshape(6, 1), ads, 4)
    for i, s in enumerate(ids):
        Wm = W + (ads[s].B @ ads[s].A if s != -1 else 0.0)
        assert np.allclose(y[i], X[i] @ Wm.T, rtol=1e-12, atol=1e-12)


def test_bad_slot_ids_are_errors():
    c = _random_case(10)
    for bad in (-2, c["S"]):
        slots = c["slots"].copy()
        slots[3, 1] = bad
        with pytest.raises(oracle.OracleError) as e:
            oracle.linear(c["x"], c["W"], slots, c["adapters"], c["S"])
        assert e.value.code == oracle.ORACLE_ERR_BAD_SLOT
    ads = dict(c["adapters"])
    ads.pop(2)
    slots = np.full_like(c["slots"], 2)
    with pytest.raises(oracle.OracleError):
        oracle.linear(c["x"], c["W"], slots, ads, c["S"])       # slot 2 never loaded


def test_threads_do_not_change_results():
    c = _random_case(11, T=33)
    y1 = oracle.linear(c["x"], c["W"], c["slots"], c["adapters"], c["S"], scales=c["scales"], threads=1)
    y8 = oracle.linear(c["x"], c["W"], c["slots"], c["adapters"], c["S"], scales=c["scales"], threads=8)
    assert np.array_equal(y1, y8)


def test_empty_batch():
    c = _random_case(12)
    y = oracle.linear(np.zeros((0, c["K"])), c["W"], np.zeros((0, 2), dtype=np.int32), c["adapters"], c["S"])
    assert y.shape == (0, c["D"])


# ----------------------------------------------------------------------------- meta
def test_meta_reproduces_the_printed_segments():
    g = dict(read_golden("segments_six_tokens.txt"))
    ids = [int(v) for v in g["ids"]]
    m = oracle.meta(np.array(ids).reshape(-1, 1))
    counts = {int(k): int(v) for k, v in (kv.split(":") for kv in g["counts"])}
    got = {s: m["seg_off"][i + 1] - m["seg_off"][i] for i, s in enumerate(m["seg_slot"])}
    assert got == counts
    assert m["order"] == [int(v) for v in g["order"]]
    assert m["seg_slot"] == [int(v) for v in g["seg_slot"]]
    assert m["seg_off"] == [int(v) for v in g["seg_off"]]
    assert m["n_active"] == int(g["n_active"][0])


@pytest.mark.parametrize("seed", range(5))
def test_meta_matches_numpy_stable_argsort(seed):
    rng = np.random.default_rng(seed)
    T, J, S = int(rng.integers(1, 300)), int(rng.integers(1, 4)), int(rng.integers(1, 130))
    ts = rng.integers(-1, S, size=(T, J))
    m = oracle.meta(ts, S)
    flat = ts.reshape(-1)
    assert m["order"] == np.argsort(flat, kind="stable").tolist()
    vals, counts = np.unique(flat, return_counts=True)
    assert m["seg_slot"] == vals.tolist()
    assert m["seg_off"] == [0] + np.cumsum(counts).tolist()
    assert m["n_active"] == int((flat != -1).sum())


def test_meta_rejects_bad_ids():
    with pytest.raises(ValueError):
        oracle.meta(np.array([[0], [5]]), 5)
    with pytest.raises(ValueError):
        oracle.meta(np.array([[-2]]), 5)


# ----------------------------------------------------------------------------- memory
def test_memory_figures_printed_by_the_page():
    GiB, MiB = 2.0 ** 30, 2.0 ** 20
    for key, v in read_golden("memory_figures.txt"):
        if key == "base_gib":
            assert round(memory.base_bytes() / GiB, int(v[1])) == float(v[0])
        elif key == "adapter_mib":
            assert round(memory.adapter_bytes(int(v[0])) / MiB, int(v[2])) == float(v[1])
        elif key == "hundred_rank16_gib":
            assert round(100 * memory.adapter_bytes(16) / GiB, int(v[1])) == float(v[0])
        elif key == "hundred_copies_gib":
            assert round(100 * memory.base_bytes() / GiB, int(v[1])) == float(v[0])
        elif key == "slots_gib":
            assert round(memory.slot_bytes(int(v[0]), int(v[1])) / GiB, int(v[3])) == float(v[2])
        elif key == "padding_numbers":
            d, r, R, small, big = map(int, v)
            assert r * (d + d) == small and R * (d + d) == big


# ----------------------------------------------------------------------------- mutation test
_MUTANTS = {
    "rslora factor uses r": ("alpha / sqrt((double)r)", "alpha / (double)r"),
    "plain factor uses sqrt": ("alpha / (double)r;", "alpha / sqrt((double)r);"),
    "scale ignored": ("const double sc = w->scales ?", "const double sc = 1.0 || w->scales ?"),
    "base term dropped": ("for (int i = 0; i < w->K; ++i) acc += Wo[i] * xt[i];", ""),
    "only first slot": ("for (int j = 0; j < w->J; ++j) {\n                const int s",
                        "for (int j = 0; j < 1; ++j) {\n                const int s"),
    "B transposed": ("const double* Bo = w->B[s] + (size_t)o * (size_t)r;", "const double* Bo = w->B[s] + (size_t)o;"),
    "A indexed by column": ("As[(size_t)q * (size_t)w->K + (size_t)i]", "As[(size_t)i * (size_t)w->rank[s] % 3 + (size_t)q]"),
    "wrong token row": ("const double* xt = w->x + (size_t)t * (size_t)w->K;",
                        "const double* xt = w->x + (size_t)(t + 1 < w->T ? t + 1 : t) * (size_t)w->K;"),
    "scale taken from slot 0 of the token": ("w->scales[(size_t)t * (size_t)w->J + (size_t)j] : 1.0",
                                             "w->scales[(size_t)t * (size_t)w->J] : 1.0"),
    "sign of side path": ("acc += c[j] * side;", "acc -= c[j] * side;"),
}


def _pins_pass(lib) -> bool:
    """The pins above, run against another build of the oracle source. True when all hold."""
    try:
        c = _hand_case()
        if not np.array_equal(oracle.linear(c["x"], c["W"], c["slots"], c["adapters"], c["S"],
                                            scales=c["scales"], lib=lib), c["y"]):
            return False
        c["adapters"][1].rslora = False
        if not np.array_equal(oracle.linear(c["x"], c["W"], c["slots"], c["adapters"], c["S"],
                                            scales=c["scales"], lib=lib), c["y_plain"]):
            return False
        r = _random_case(4, J=1)
        ad = r["adapters"][1]
        y = oracle.linear(r["x"], r["W"], np.full((r["T"], 1), 1), r["adapters"], r["S"], lib=lib)
        ym = r["x"] @ (r["W"] + _factor(ad) * (ad.B @ ad.A)).T
        return bool(np.max(np.abs(y - ym)) <= 1e-12 * np.max(np.abs(ym)))
    except Exception:
        return False


def _pins_pass_in_child(lib_path: str) -> bool:
    """Run the pins on a mutant in a child process: a mutant that crashes counts as caught."""
    import sys
    code = ("import sys; sys.path[:0] = [%r]; import oracle; from tests import test_oracle as t; "
            "sys.exit(0 if t._pins_pass(oracle.load_library(%r)) else 3)") % (
                os.path.dirname(os.path.dirname(os.path.abspath(__file__))), lib_path)
    rc = subprocess.run([sys.executable, "-c", code], capture_output=True, timeout=120).returncode
    return rc == 0


def test_pins_catch_planted_mistakes():
    if shutil.which("gcc") is None:
        pytest.skip("gcc missing")
    src = open(oracle._SRC).read()
    assert _pins_pass(oracle.load_library())
    with tempfile.TemporaryDirectory() as tmp:
        for i, (name, (old, new)) in enumerate(_MUTANTS.items()):
            assert old in src, f"mutation '{name}' no longer applies to the oracle source"
            msrc = os.path.join(tmp, f"mutant{i}.c")
            with open(msrc, "w") as f:
                f.write(src.replace(old, new, 1))
            lib_path = os.path.join(tmp, f"mutant{i}.so")
            oracle.compile_library(msrc, lib_path, force=True)   # every mutant must compile
            assert not _pins_pass_in_child(lib_path), f"pins missed mutant: {name}"
