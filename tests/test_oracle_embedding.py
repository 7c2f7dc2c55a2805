"""Pins for the embedding oracle (oracle/embed.py): a hand-worked example, the one-hot
identity against the linear-layer oracle (separate C code), exact sentinel rows, the merged
table, the error cases, and planted mistakes in the oracle's source that the pins must catch."""
import os
import types
from types import SimpleNamespace

import numpy as np
import pytest

import oracle
from oracle import embed as emb_mod
from tests.conftest import read_golden


def _hand_case():
    d, slots = {}, {}
    for key, vals in read_golden("embedding_hand.txt"):
        if key == "slot":
            kv = dict(zip(vals[1::2], vals[2::2]))
            slots[int(vals[0])] = SimpleNamespace(rank=int(kv["rank"]), alpha=float(kv["alpha"]),
                                                  rslora=bool(int(kv["rslora"])))
        else:
            d[key] = vals
    V, D, J, S = (int(d[k][0]) for k in ("V", "D", "J", "n_slots"))
    f = lambda k: np.array([float(v) for v in d[k]])  # noqa: E731
    for s, ad in slots.items():
        ad.A = f(f"A{s}").reshape(ad.rank, V)
        ad.B = f(f"B{s}").reshape(D, ad.rank)
    ids = np.array([int(v) for v in d["ids"]])
    T = len(ids)
    return dict(V=V, D=D, J=J, S=S, T=T, E=f("E").reshape(V, D), ids=ids, adapters=slots,
                slots=np.array([int(v) for v in d["token_slots"]]).reshape(T, J),
                scales=f("scales").reshape(T, J), y=f("y").reshape(T, D), y_plain=f("y_plain").reshape(T, D))


def _random_case(seed, T=9, V=23, D=14, J=2, S=4, ranks=(3, 5, 2, 4)):
    rng = np.random.default_rng(seed)
    ads = {s: SimpleNamespace(A=rng.standard_normal((ranks[s], V)), B=rng.standard_normal((D, ranks[s])),
                              rank=ranks[s], alpha=float(rng.integers(1, 9)), rslora=bool(s % 2))
           for s in range(S)}
    return dict(V=V, D=D, J=J, S=S, T=T, E=rng.standard_normal((V, D)), ids=rng.integers(0, V, size=T),
                slots=rng.integers(-1, S, size=(T, J)), scales=rng.uniform(0.2, 1.0, size=(T, J)), adapters=ads)


def _run(c, fn=None, **kw):
    fn = fn or emb_mod.embedding
    return fn(c["ids"], c["E"], c["slots"], c["adapters"], c["S"], scales=c["scales"], **kw)


def _one_hot_linear(c):
    """The same lookup through the linear-layer oracle: x = one-hot rows of the ids, W = E^T."""
    x = np.zeros((c["T"], c["V"]))
    x[np.arange(c["T"]), c["ids"]] = 1.0
    return oracle.linear(x, c["E"].T, c["slots"], c["adapters"], c["S"], scales=c["scales"])


def _close(a, b, tol=1e-12):
    return float(np.max(np.abs(a - b))) <= tol * max(1.0, float(np.max(np.abs(b))))


# ----------------------------------------------------------------------------- pins
def test_hand_example_plain_and_rslora():
    c = _hand_case()
    assert np.array_equal(_run(c), c["y"])
    c["adapters"][1].rslora = False
    assert np.array_equal(_run(c), c["y_plain"])


@pytest.mark.parametrize("seed,J", [(1, 1), (2, 2), (3, 3), (4, 8)])
def test_lookup_equals_the_linear_layer_on_one_hot_inputs(seed, J):
    c = _random_case(seed, J=J)
    assert _close(_run(c), _one_hot_linear(c))


def test_sentinel_rows_are_the_table_rows_exactly():
    c = _random_case(5, T=12, J=3)
    c["slots"][::3] = -1
    y = _run(c)
    for t in range(0, c["T"], 3):
        assert np.array_equal(y[t], c["E"][c["ids"][t]])


@pytest.mark.parametrize("rslora", [False, True])
def test_single_adapter_equals_the_merged_table(rslora):
    c = _random_case(6, T=15, J=1)
    ad = c["adapters"][2]
    ad.rslora = rslora
    c["slots"][:] = 2
    c["scales"][:] = 0.75
    factor = ad.alpha / (np.sqrt(ad.rank) if rslora else ad.rank)
    merged = c["E"] + 0.75 * factor * (ad.B @ ad.A).T           # [V, D]
    assert _close(_run(c), merged[c["ids"]])


def test_row_selection_and_empty_batch():
    c = _random_case(7, T=10)
    rows = np.array([9, 0, 4])
    assert np.array_equal(_run(c, rows=rows), _run(c)[rows])
    e = dict(c, T=0, ids=np.zeros(0, np.int64), slots=np.zeros((0, 2), np.int64), scales=np.zeros((0, 2)))
    assert _run(e).shape == (0, c["D"])


def test_bad_ids_and_slots_are_errors():
    c = _random_case(8)
    for bad in (-1, c["V"]):
        d = dict(c, ids=c["ids"].copy())
        d["ids"][3] = bad
        with pytest.raises(oracle.OracleError):
            _run(d)
    for bad in (-2, c["S"]):
        d = dict(c, slots=c["slots"].copy())
        d["slots"][2, 0] = bad
        with pytest.raises(oracle.OracleError):
            _run(d)
    d = dict(c, adapters={s: a for s, a in c["adapters"].items() if s != 1}, slots=np.full_like(c["slots"], 1))
    with pytest.raises(oracle.OracleError):
        _run(d)


# ----------------------------------------------------------------------------- mutation test
_MUTANTS = {
    "rsLoRA factor uses r": ("np.sqrt(float(ad.rank)) if ad.rslora else float(ad.rank)",
                             "float(ad.rank) if ad.rslora else float(ad.rank)"),
    "plain factor uses sqrt": ("np.sqrt(float(ad.rank)) if ad.rslora else float(ad.rank)",
                               "np.sqrt(float(ad.rank)) if ad.rslora else np.sqrt(float(ad.rank))"),
    "table row dropped": ("acc = _f64(E[i]).copy()", "acc = np.zeros(D)"),
    "wrong table row": ("acc = _f64(E[i]).copy()", "acc = _f64(E[(i + 1) % V]).copy()"),
    "column of the next id": ("a_col = _f64(A[:, i])", "a_col = _f64(A[:, (i + 1) % V])"),
    "scale ignored": ("(1.0 if sc is None else float(sc[t, j]))", "1.0"),
    "scale of the token's first slot": ("float(sc[t, j])", "float(sc[t, 0])"),
    "only the first slot": ("for j in range(J):", "for j in range(1):"),
    "side path subtracted": ("acc += (1.0", "acc -= (1.0"),
    "B rows reversed": ("side = B64[s] @ a_col", "side = B64[s][::-1] @ a_col"),
}


def _pins_pass(fn) -> bool:
    try:
        c = _hand_case()
        if not np.array_equal(_run(c, fn), c["y"]):
            return False
        c["adapters"][1].rslora = False
        if not np.array_equal(_run(c, fn), c["y_plain"]):
            return False
        r = _random_case(11, J=3)
        return _close(_run(r, fn), _one_hot_linear(r))
    except Exception:
        return False


def test_pins_catch_planted_mistakes():
    src = open(emb_mod.__file__).read()
    assert _pins_pass(emb_mod.embedding)
    for name, (old, new) in _MUTANTS.items():
        assert old in src, f"mutation '{name}' no longer applies to the oracle source"
        mod = types.ModuleType("oracle._embedding_mutant")
        mod.__package__ = "oracle"
        mod.__file__ = os.devnull
        exec(compile(src.replace(old, new, 1), f"<mutant {name}>", "exec"), mod.__dict__)
        assert not _pins_pass(mod.embedding), f"pins missed mutant: {name}"
