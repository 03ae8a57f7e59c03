"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in a copy of an oracle module: the module's
source with one text substitution, loaded as a separate module object; the
oracle package itself is never modified.  Then it runs that module's pin suite
(every test of the pin file, every parameter set) with the copy in place of the
oracle and checks that at least one pin fails.  The unmodified source must pass
the same harness, so a failure can only come from the planted mistake.
"""

from __future__ import annotations

import itertools
import pathlib
import types

import pytest

import test_oracle_attention as attention_pins
import test_oracle_fp8 as fp8_pins
import test_oracle_metadata as metadata_pins

ORACLE = pathlib.Path(__file__).resolve().parent.parent / "oracle"

# (pin module, attribute the pins call the oracle through, oracle source file)
SUITES = {
    "attention": (attention_pins, "oa", ORACLE / "attention.py"),
    "metadata": (metadata_pins, "om", ORACLE / "metadata.py"),
    "fp8": (fp8_pins, "fp8", ORACLE / "fp8.py"),
}

# name -> (suite, text in the oracle source, replacement): one plausible mistake each
MUTANTS = {
    # attention
    "gqa_head_modulo": ("attention", "g = h // group", "g = h % Hkv"),
    "scale_dropped": ("attention", "scores = scale * (q_rows @ keys.T)", "scores = q_rows @ keys.T"),
    "block_index_by_offset": ("attention", "block_table[t // block_size]", "block_table[t % block_size]"),
    "offset_shifted": ("attention", "cache[block, t % block_size]", "cache[block, (t + 1) % block_size]"),
    "context_short_by_one": ("attention", "block_tables[b], ctx)", "block_tables[b], ctx - 1)"),
    "values_from_k_cache": ("attention", "values = gather_tokens(v_cache,", "values = gather_tokens(k_cache,"),
    "softmax_not_normalised": ("attention", "return (p @ values) / p.sum(axis=1, keepdims=True)",
                               "return p @ values"),
    "causal_top_left": ("attention", "visible = cols <= cached + rows", "visible = cols <= rows"),
    "causal_strict": ("attention", "visible = cols <= cached + rows", "visible = cols < cached + rows"),
    "history_short_by_one": ("attention", "cached = nk - nq", "cached = nk - nq - 1"),
    "non_causal_still_masked": ("attention", "if causal:", "if True:"),
    "packed_keys_at_query_offsets": ("attention", "keys = _f64(k[k0:k1])", "keys = _f64(k[q0:q0 + nk])"),
    "combine_l_unweighted": ("attention", "total_l = sum(w[j] * parts[j][2]", "total_l = sum(parts[j][2]"),
    "combine_weights_inverted": ("attention", "w = np.exp(ms - big_m)", "w = np.exp(big_m - ms)"),
    "partial_o_normalised": ("attention", "o[h] = p @ values[lo:hi, g]", "o[h] = p @ values[lo:hi, g] / p.sum()"),
    "store_block_offset_swapped": ("attention", "block, offset = divmod(slot, block_size)",
                                   "offset, block = divmod(slot, block_size)"),
    "store_padding_not_skipped": ("attention", "if slot == -1:\n            continue",
                                  "if slot < -1:\n            continue"),
    "copy_direction_reversed": ("attention", "c[dst] = orig[src]", "c[src] = orig[dst]"),
    # metadata
    "blocks_needed_one_extra": ("metadata", "while covered < num_tokens:", "while covered <= num_tokens:"),
    "append_rule_shifted": ("metadata", "return length % block_size == 0", "return length % block_size == 1"),
    "slot_block_not_scaled": ("metadata", "slot_mapping.append(block_id * block_size + i % block_size)",
                              "slot_mapping.append(block_id + i % block_size)"),
    "cu_k_counts_new_tokens_only": ("metadata", "cu_k.append(cu_k[-1] + end)",
                                    "cu_k.append(cu_k[-1] + end - start)"),
    "tables_always_needed": ("metadata", "need_tables = cu_k[-1] > cu_q[-1]", "need_tables = cu_k[-1] >= cu_q[-1]"),
    "decode_slot_one_past": ("metadata", "table[-1] * block_size + last_block_num_tokens - 1",
                             "table[-1] * block_size + last_block_num_tokens"),
    "context_excludes_new_token": ("metadata", "context_lens.append(length)", "context_lens.append(length - 1)"),
    "positions_restart_at_zero": ("metadata", "positions.extend(range(start, end))",
                                  "positions.extend(range(0, end - start))"),
    # fp8
    "exponent_bias_8": ("fp8", "np.power(2.0, exp - 7)", "np.power(2.0, exp - 8)"),
    "subnormal_scale": ("fp8", "sub = mant / 8.0 * 2.0 ** -6", "sub = mant / 8.0 * 2.0 ** -7"),
    "ties_not_to_even": ("fp8", "((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0) & (hi != lo))",
                         "((d_hi == d_lo) & (hi != lo))"),
    "sign_dropped": ("fp8", "code = np.where(neg, code | 0x80, code)", "code = np.where(neg, code, code)"),
    "fp8_store_v_with_k_scale": ("fp8", "quantize(v[i], v_scale)", "quantize(v[i], k_scale)"),
    "fp8_store_block_offset_swapped": ("fp8", "blk, off = divmod(slot, bs)", "off, blk = divmod(slot, bs)"),
    "quantize_divides_in_float64": ("fp8", "q = np.asarray(x, dtype=np.float32) / np.float32(scale)",
                                    "q = np.asarray(x, dtype=np.float64) / float(scale)"),
}


def _load(path: pathlib.Path, old: str | None = None, new: str | None = None) -> types.ModuleType:
    src = path.read_text()
    if old is not None:
        assert old in src, f"mutation site not found in {path.name}: {old!r}"
        src = src.replace(old, new)
    mod = types.ModuleType(f"oracle_copy_{path.stem}")
    exec(compile(src, str(path), "exec"), mod.__dict__)
    return mod


def _cases(fn):
    """Every argument set the function's parametrize marks give (one empty set if none)."""
    combos = [{}]
    for mark in getattr(fn, "pytestmark", []):
        if mark.name != "parametrize":
            continue
        names = mark.args[0]
        names = [n.strip() for n in names.split(",")] if isinstance(names, str) else list(names)
        expanded = []
        for base, values in itertools.product(combos, mark.args[1]):
            values = values if len(names) > 1 else (values,)
            expanded.append({**base, **dict(zip(names, values))})
        combos = expanded
    return combos


def _pins(module):
    return [getattr(module, n) for n in sorted(dir(module)) if n.startswith("test_") and callable(getattr(module, n))]


def _first_failure(suite: str, oracle_copy: types.ModuleType, monkeypatch) -> str | None:
    """Runs the suite's pins against `oracle_copy`; returns the first failing pin, or None."""
    pins, attr, _ = SUITES[suite]
    monkeypatch.setattr(pins, attr, oracle_copy)
    for fn in _pins(pins):
        for kwargs in _cases(fn):
            try:
                fn(**kwargs)
            except Exception:  # an assertion or an error raised by the planted mistake
                return f"{fn.__name__}({kwargs})"
    return None


@pytest.mark.parametrize("suite", sorted(SUITES))
def test_unmodified_oracle_passes_the_harness(suite, monkeypatch):
    pins, _, path = SUITES[suite]
    assert len(_pins(pins)) >= 6
    assert _first_failure(suite, _load(path), monkeypatch) is None


@pytest.mark.filterwarnings("ignore::RuntimeWarning")  # some mistakes produce NaN rows
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(name, monkeypatch):
    suite, old, new = MUTANTS[name]
    failed = _first_failure(suite, _load(SUITES[suite][2], old, new), monkeypatch)
    assert failed is not None, f"no pin catches the planted mistake {name!r}"
