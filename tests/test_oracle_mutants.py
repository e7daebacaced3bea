"""Planted mistakes in the oracle must each fail at least one pin.

Each case rewrites one line of an oracle module's source (a dropped term, a
wrong sign, bound or index, a transposed operand, sigma used where sigma^-1
belongs), loads the rewritten module, rebinds its functions wherever the
oracle holds them, and runs the pins of ``test_oracle_pins`` (all but the
slow receptive-field statistics).  A mutant that every pin accepts is a
mistake the pins could not see.  Everything runs on the CPU; nothing here
touches the CUDA path.
"""

from __future__ import annotations

import inspect
import re
import time
import types

import pytest

import oracle
from oracle import attention, graph, prng

import test_oracle_pins as pins

MODULES = {"prng": prng, "graph": graph, "attention": attention}

# (id, module, original text, planted text)
MUTANTS = [
    ("splitmix-shift", "prng", "z = ((z ^ (z >> 30)) * MIX1) & MASK64",
     "z = ((z ^ (z >> 31)) * MIX1) & MASK64"),
    ("splitmix-gamma", "prng", "state = (state + GOLDEN_GAMMA) & MASK64",
     "state = (state + GOLDEN_GAMMA + 2) & MASK64"),
    ("stream-ignores-layer", "prng", "start = (seed + (layer << 32) + batch_index) & MASK64",
     "start = (seed + batch_index) & MASK64"),
    ("stream-layer-shift", "prng", "start = (seed + (layer << 32) + batch_index) & MASK64",
     "start = (seed + (layer << 31) + batch_index) & MASK64"),
    ("stream-without-mixing-step", "prng", "    _, out = splitmix64_step(start)\n",
     "    out = start\n"),
    ("draws-state-not-output", "prng", "        return out\n\n    return fisher_yates(n, draw)",
     "        return state\n\n    return fisher_yates(n, draw)"),
    ("sattolo-draw", "prng", "j = (x * (i + 1)) >> 64", "j = (x * i) >> 64"),
    ("shuffle-skips-last", "prng", "for i in range(n - 1, 0, -1):",
     "for i in range(n - 2, 0, -1):"),
    ("inverse-is-sigma", "prng", "inv[b, i] = p", "inv[b, p] = i"),
    ("window-right-short", "graph", "lo, hi = max(0, p - h), min(n - 1, p + h)",
     "lo, hi = max(0, p - h), min(n - 1, p + h - 1)"),
    ("window-left-short", "graph", "lo, hi = max(0, p - h), min(n - 1, p + h)",
     "lo, hi = max(0, p - h + 1), min(n - 1, p + h)"),
    ("window-wraps", "graph", "keys = [int(perm[q]) for q in range(lo, hi + 1)]",
     "keys = sorted({int(perm[q % n]) for q in range(p - h, p + h + 1)})"),
    ("sigma-for-inverse", "graph", "p = int(inv[i])", "p = int(perm[i])"),
    ("causal-drops-self", "graph", "keys = [j for j in keys if j <= i]",
     "keys = [j for j in keys if j < i] or [i]"),
    ("causal-flipped", "graph", "keys = [j for j in keys if j <= i]",
     "keys = [j for j in keys if j >= i]"),
    ("half-width-ceil", "graph", "return window // 2", "return (window + 1) // 2"),
    ("swa-extra-key", "graph", "return np.arange(max(0, i - window + 1), i + 1, dtype=np.int64)",
     "return np.arange(max(0, i - window), i + 1, dtype=np.int64)"),
    ("pairs-noncausal-halved", "graph", "return n + (far if causal else 2 * far)",
     "return n + far"),
    ("pair-probability-term", "graph", "return (2 * h * n - h * (h + 1)) / (n * (n - 1))",
     "return (2 * h * n - h * h) / (n * (n - 1))"),
    ("receptive-field-layer-order", "graph",
     "reach = (a.astype(np.int64) @ reach.astype(np.int64)) > 0",
     "reach = (reach.astype(np.int64) @ a.astype(np.int64)) > 0"),
    ("scale-dropped", "attention", 's = scale * np.einsum("hd,mhd->hm", qrow, kh)',
     's = np.einsum("hd,mhd->hm", qrow, kh)'),
    ("k-for-v", "attention", "vh = vb[keys][:, head_map, :]", "vh = kb[keys][:, head_map, :]"),
    ("gqa-head-modulo", "attention", "return np.arange(hq) // (hq // hkv)",
     "return np.arange(hq) % hkv"),
    ("softmax-normalised-over-heads", "attention", "p = e / e.sum(axis=1, keepdims=True)",
     "p = e / e.sum(axis=0, keepdims=True)"),
    ("gates-swapped", "attention", "return g1 * y_sa + g2 * y_swa",
     "return g2 * y_sa + g1 * y_swa"),
    ("swa-window-zero-taken-literally", "attention",
     "w_swa = window if (window_swa is None or window_swa <= 0) else window_swa",
     "w_swa = window if (window_swa is None or window_swa < 0) else window_swa"),
    ("swa-window-ignored", "attention",
     "w_swa = window if (window_swa is None or window_swa <= 0) else window_swa",
     "w_swa = window"),
    ("sigmoid-sign", "attention", "return 1.0 / (1.0 + np.exp(-x))",
     "return 1.0 / (1.0 + np.exp(x))"),
    ("sigmoid-slope", "attention", "return 1.0 / (1.0 + np.exp(-x))",
     "return 1.0 / (1.0 + np.exp(-2.0 * x))"),
    ("mask-fills-zero", "attention", "s = np.where(mask, s, -np.inf)",
     "s = np.where(mask, s, 0.0)"),
    ("causal-full-upper", "attention",
     "mask = np.tril(np.ones((n, n), dtype=bool)) if causal",
     "mask = np.triu(np.ones((n, n), dtype=bool)) if causal"),
]

# The pins, with the arguments of their parametrised forms.
PINS = [
    ("splitmix64 vectors", pins.test_splitmix64_published_vectors, ()),
    ("Fisher-Yates stub draws", pins.test_fisher_yates_index_mapping_with_stub_draws, ()),
    ("uniform over S4", pins.test_perm_draw_is_uniform_over_s4, ()),
    ("streams differ", pins.test_streams_differ_by_layer_and_batch, ()),
    ("stream state", pins.test_stream_state_is_one_published_step_from_the_start, ()),
    ("make_perm wiring", pins.test_make_perm_consumes_successive_stream_outputs, ()),
    ("inverse", pins.test_inverse_perm, ()),
    ("hand sets w=2", pins.test_hand_worked_neighbour_sets, ("sa_hand_n6.txt",)),
    ("hand sets w=5", pins.test_hand_worked_neighbour_sets, ("sa_hand_n6_w5.txt",)),
    ("pair count nc", pins.test_attended_pair_count_closed_form, (17, 4, False)),
    ("pair count c", pins.test_attended_pair_count_closed_form, (64, 9, True)),
    ("pair count clipped nc", pins.test_attended_pair_count_closed_form, (64, 200, False)),
    ("pair count clipped c", pins.test_attended_pair_count_closed_form, (64, 200, True)),
    ("pair count w=1", pins.test_attended_pair_count_closed_form, (33, 1, False)),
    ("closed forms at full windows", pins.test_closed_forms_at_full_windows, ()),
    ("expected degree", pins.test_expected_degree_closed_form, ()),
    ("pair probability", pins.test_pair_probability_matches_closed_form_and_w_over_n, ()),
    ("SWA receptive field", pins.test_receptive_field_swa_is_linear, ()),
    ("receptive field by set unions", pins.test_receptive_field_matches_set_unions_over_layers, ()),
    ("full attention nc", pins.test_full_attention_matches_sdpa, (False,)),
    ("full attention c", pins.test_full_attention_matches_sdpa, (True,)),
    ("identity sigma", pins.test_identity_perm_is_banded_attention, ()),
    ("SWA vs SDPA", pins.test_swa_matches_masked_sdpa, ()),
    ("wide window", pins.test_wide_window_is_full_attention, ()),
    ("permuted route nc", pins.test_permuted_space_route_agrees, (False,)),
    ("permuted route c", pins.test_permuted_space_route_agrees, (True,)),
    ("relabelling", pins.test_relabelling_equivariance_noncausal, ()),
    ("gate limits", pins.test_gate_limits_reduce_to_single_paths, ()),
    ("gated SWA window", pins.test_gated_swa_window_is_its_own, ()),
    ("gated logistic", pins.test_gated_merge_with_arbitrary_logits_uses_the_logistic_function, ()),
    ("GQA and scale", pins.test_gqa_head_map_and_scale_pinned_by_sdpa, ()),
    ("large scores", pins.test_softmax_is_stable_at_large_scores, ()),
    ("argument checks", pins.test_argument_checks, ()),
]


def _plant(monkeypatch, modname: str, old: str, new: str) -> None:
    """Load ``oracle.<modname>`` with ``old`` replaced by ``new`` and rebind
    each of its functions in every oracle module that holds it."""
    mod = MODULES[modname]
    src = inspect.getsource(mod)
    assert src.count(old) == 1, f"mutation site not found once in oracle.{modname}: {old!r}"
    mutant = types.ModuleType(f"{mod.__name__}_mutant")
    mutant.__package__ = "oracle"
    mutant.__file__ = mod.__file__
    exec(compile(src.replace(old, new), mod.__file__, "exec"), mutant.__dict__)
    for name, fn in list(vars(mod).items()):
        if inspect.isfunction(fn) and fn.__module__ == mod.__name__:
            for holder in (oracle, prng, graph, attention):
                if getattr(holder, name, None) is fn:
                    monkeypatch.setattr(holder, name, mutant.__dict__[name])


def _caught_by(deadline: float) -> list[str]:
    caught = []
    for name, fn, args in PINS:
        try:
            fn(*args)
        except pytest.skip.Exception:
            continue  # a pin whose library is missing here decides nothing
        except (Exception, pytest.fail.Exception):  # an assertion, pytest.raises
            caught.append(name)                     # not raising, or a broken
            break                                   # precondition: one is enough
        if time.monotonic() > deadline:
            break
    return caught


def test_unmutated_oracle_passes_every_pin():
    for name, fn, args in PINS:
        fn(*args)


@pytest.mark.parametrize("modname,old,new", [
    ("attention", "p = e / e.sum(axis=1, keepdims=True)",
     "p = e / (1.0 * e.sum(axis=1, keepdims=True))"),
    ("graph", "return window // 2", "return (2 * window) // 4"),
    ("prng", "j = (x * (i + 1)) >> 64", "j = (x * i + x) >> 64"),
])
def test_equivalent_rewrite_passes_every_pin(monkeypatch, modname, old, new):
    """Control: planting a rewrite that changes nothing must not trip a pin,
    so a caught mutant is caught for its mistake, not for being planted."""
    _plant(monkeypatch, modname, old, new)
    for name, fn, args in PINS:
        fn(*args)


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("mid,modname,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(monkeypatch, mid, modname, old, new):
    _plant(monkeypatch, modname, old, new)
    caught = _caught_by(time.monotonic() + 60.0)
    assert caught, f"no pin detects the planted mistake {mid!r} in oracle.{modname}"


# ------------------------------------------------------- single-operator scan
# Every single-token change of the kinds below, on every code line of the
# oracle modules, must fail a pin -- except these, which compute the same
# values (module, original line, mutated line, why):
EQUIVALENT = {
    ("graph", "h = min(half_width(window), n - 1) if n > 0 else 0",
     "h = min(half_width(window), n - 1) if n >= 0 else 0"): "n = 0 gives 0 pairs either way",
    ("graph", "h = min(half_width(window), n - 1) if n > 0 else 0",
     "h = min(half_width(window), n - 0) if n > 0 else 0"): "the extra distance d = n adds n - n = 0",
    ("graph", "return w * (w + 1) // 2 + (n - w) * w",
     "return w * (w + 1) / 2 + (n - w) * w"): "w(w+1) is even: the same value, as a float",
    ("graph", "h = min(half_width(window), n - 1)",
     "h = min(half_width(window), n - 0)"): "h = n and h = n - 1 give the same closed form",
    ("attention", "causal: bool = True, scale: float | None = None, rows=None) -> np.ndarray:",
     "causal: bool = False, scale: float | None = None, rows=None) -> np.ndarray:"):
        "a default that every caller overrides",
}
SWAPS = [(r"<=", "<"), (r"(?<![<>=!])<(?![<=])", "<="), (r">=", ">"),
         (r"(?<![<>=\-])>(?![>=])", ">="), (r" \+ ", " - "), (r" - ", " + "), (r"//", "/"),
         (r"\+ 1\b", "+ 2"), (r"- 1\b", "- 2"), (r"\b1\b", "0"), (r"\b2\b", "3"),
         (r"\*\*", "*"), (r"axis=1", "axis=0"), (r"\bTrue\b", "False")]
SKIP_PREFIXES = ("#", '"""', "def ", "raise", "from ", "import ")


def _single_operator_mutants():
    for modname, mod in MODULES.items():
        lines = inspect.getsource(mod).split("\n")
        in_doc = False
        for li, line in enumerate(lines):
            st = line.strip()
            if st.count('"""') == 1:
                in_doc = not in_doc
                continue
            if in_doc or not st or st.startswith(SKIP_PREFIXES):
                continue
            code = line.split("#")[0]
            for pat, rep in SWAPS:
                for m in re.finditer(pat, code):
                    new = code[:m.start()] + re.sub(pat, rep, code[m.start():m.end()]) + code[m.end():]
                    if new != code:
                        yield modname, li, code, new


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
def test_every_single_operator_mutant_fails_a_pin_or_is_equivalent(monkeypatch):
    survivors, count = [], 0
    for modname, li, code, new in _single_operator_mutants():
        mod = MODULES[modname]
        lines = inspect.getsource(mod).split("\n")
        src = "\n".join(lines[:li] + [new] + lines[li + 1:])
        mutant = types.ModuleType(f"{mod.__name__}_mutant")
        mutant.__package__ = "oracle"
        mutant.__file__ = mod.__file__
        try:
            exec(compile(src, mod.__file__, "exec"), mutant.__dict__)
        except Exception:
            continue  # not valid Python: not a mutant
        count += 1
        with monkeypatch.context() as mp:
            for name, fn in list(vars(mod).items()):
                if inspect.isfunction(fn) and fn.__module__ == mod.__name__:
                    for holder in (oracle, prng, graph, attention):
                        if getattr(holder, name, None) is fn:
                            mp.setattr(holder, name, mutant.__dict__[name])
            caught = _caught_by(time.monotonic() + 60.0)
        if not caught and (modname, code.strip(), new.strip()) not in EQUIVALENT:
            survivors.append(f"oracle.{modname} line {li + 1}: {code.strip()!r} -> {new.strip()!r}")
    assert count > 100
    assert not survivors, "mutants no pin rejects:\n" + "\n".join(survivors)
