"""Plants plausible mistakes in the CPU oracle (on the CPU only) and checks that
at least one pin from ``oracle_pins`` fails for each of them."""
import numpy as np
import pytest

import oracle.attention_fp64 as orc
import oracle_pins

_real_visible = orc.visible_keys
_real_gather = orc.gather_kv
_real_attend = orc.softmax_attend
_real_e4m3 = orc.decode_e4m3fn


def _visible_minus_one(S, L, t):
    return max(0, min(S, S - L + t))


def _visible_plus_one(S, L, t):
    return max(0, min(S, S - L + t + 2))


def _visible_no_mask(S, L, t):
    return S


def _visible_top_left(S, L, t):
    return min(S, t + 1)


def _head_modulo(h, group, num_kv_heads):
    return h % num_kv_heads


def _gather_logical_pages(cache_raw, decode, row, S, descale, start=0):
    return _real_gather(cache_raw, decode, np.arange(len(row)), S, descale, start)


def _gather_no_descale(cache_raw, decode, row, S, descale, start=0):
    return _real_gather(cache_raw, decode, row, S, 1.0, start)


def _attend_no_scale(q, K, V, n, scale, *rest):
    return _real_attend(q, K, V, n, 1.0, *rest)


def _attend_abs_scale(q, K, V, n, scale, *rest):
    return _real_attend(q, K, V, n, abs(scale), *rest)


def _attend_zero_scale_as_one(q, K, V, n, scale, *rest):
    return _real_attend(q, K, V, n, scale if scale != 0 else 1.0, *rest)


def _attend_keys_as_values(q, K, V, n, scale, *rest):
    return _real_attend(q, K, K, n, scale, *rest)


def _attend_reversed_rows(q, K, V, n, scale, *rest):
    return _real_attend(q[::-1], K, V, n, scale, *rest)[::-1]


def _window_off_by_one(S, L, t, window_left):
    return 0 if window_left < 0 else max(0, S - L + t - window_left + 1)


def _window_ignored(S, L, t, window_left):
    return 0


def _no_softcap(logits, softcap):
    return logits


def _sink_ignored(sink, m):
    return 0.0 * m


def _e4m3_bias8(raw):
    return _real_e4m3(raw) * 0.5


def _e4m3_no_subnormals(raw):
    v = _real_e4m3(raw)
    r = np.asarray(raw, dtype=np.uint8)
    return np.where(((r >> 3) & 0xF) == 0, 0.0, v)


MUTATIONS = {
    "mask_off_by_minus_one": ("visible_keys", _visible_minus_one),
    "mask_off_by_plus_one": ("visible_keys", _visible_plus_one),
    "no_causal_mask": ("visible_keys", _visible_no_mask),
    "top_left_causal": ("visible_keys", _visible_top_left),
    "head_mapping_modulo": ("kv_head_of", _head_modulo),
    "ignores_block_table": ("gather_kv", _gather_logical_pages),
    "drops_descale": ("gather_kv", _gather_no_descale),
    "drops_softmax_scale": ("softmax_attend", _attend_no_scale),
    "softmax_scale_sign_dropped": ("softmax_attend", _attend_abs_scale),
    "zero_softmax_scale_as_one": ("softmax_attend", _attend_zero_scale_as_one),
    "keys_used_as_values": ("softmax_attend", _attend_keys_as_values),
    "rows_reversed": ("softmax_attend", _attend_reversed_rows),
    "window_off_by_one": ("first_visible_key", _window_off_by_one),
    "window_ignored": ("first_visible_key", _window_ignored),
    "softcap_dropped": ("softcapped", _no_softcap),
    "sink_ignored": ("sink_weight", _sink_ignored),
}

DECODER_MUTATIONS = {
    "e4m3_wrong_bias": _e4m3_bias8,
    "e4m3_flushes_subnormals": _e4m3_no_subnormals,
}


def _some_pin_fails():
    failures = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            failures.append(pin.__name__)
    return failures


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(orc, attr, fn)
    assert _some_pin_fails(), f"planted mistake {name} passed every pin"


@pytest.mark.parametrize("name", sorted(DECODER_MUTATIONS))
def test_decoder_mutation_is_caught(name, monkeypatch):
    fn = DECODER_MUTATIONS[name]
    monkeypatch.setattr(orc, "decode_e4m3fn", fn)
    monkeypatch.setitem(orc.DECODERS, "fp8_e4m3", fn)
    assert _some_pin_fails(), f"planted mistake {name} passed every pin"
