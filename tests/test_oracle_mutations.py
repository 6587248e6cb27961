"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins catch each one.

A pin set that still passes with a mistake planted is too weak to trust the
oracle with; every mutation below must make at least one pin fail.
"""

import numpy as np
import pytest

from oracle import attention as A
from oracle import fp8 as F
from oracle import metadata as M
from tests import test_oracle_pins as P

CHECKS = [
    ("bruteforce", lambda: P.check_bruteforce()),
    ("bruteforce_window", lambda: P.check_bruteforce(window=3)),
    ("sdpa", lambda: P.check_sdpa()),
    ("sdpa_window", lambda: P.check_sdpa(window=5)),
    ("single_key", P.check_single_key),
    ("uniform", P.check_uniform_scores),
    ("merge", P.check_merge_closed_form),
    ("bruteforce_noncausal", lambda: P.check_bruteforce(causal=False)),
    ("sdpa_noncausal", lambda: P.check_sdpa(causal=False)),
    ("prefix_suffix_merge", P.check_prefix_suffix_merge),
    ("ragged_bruteforce", P.check_ragged_bruteforce),
    ("ragged_bruteforce_noncausal", lambda: P.check_ragged_bruteforce(causal=False)),
    ("ragged_sdpa", P.check_ragged_sdpa),
    ("cascade", P.check_cascade_shared_prefix),
]


def _all_pins_pass():
    for _, fn in CHECKS:
        try:
            if not fn():
                return False
        except Exception:
            return False
    return True


def test_unmutated_oracle_passes_every_pin():
    assert _all_pins_pass()


MUTATIONS = {
    # GQA: interleaved instead of contiguous head groups
    "gqa_interleaved": ("kv_head_of", lambda h, group: h % 2),
    # causal alignment off by one in either direction
    "causal_plus_one": ("query_position", lambda L, n, t: L - n + t + 1),
    "causal_minus_one": ("query_position", lambda L, n, t: max(0, L - n + t - 1)),
    # top-left instead of bottom-right aligned causal mask
    "causal_top_left": ("query_position", lambda L, n, t: t),
    # window keeps w keys instead of w + 1
    "window_w_keys": ("visible_range", lambda p, w: ((0 if w < 0 else max(0, p - w + 1)), p)),
    # ignore last_page_len: treat the last page as full
    "full_last_page": ("kv_len_of", lambda n, last, ps: n * ps),
    # last page length off by one
    "last_page_off_by_one": ("kv_len_of", lambda n, last, ps: 0 if n == 0 else (n - 1) * ps + last - 1),
    # gather by offset only within the first page
    "gather_ignores_pages": ("gather_logical", lambda pool, pages, L, ps: pool[np.asarray(pages)[np.zeros(L, dtype=np.int64)], np.arange(L) % ps]),
    # non-causal range loses its last key, or its first
    "noncausal_drops_last": ("full_range", lambda L: (0, L - 2)),
    "noncausal_from_one": ("full_range", lambda L: (1, L - 1)),
    # ragged K/V rows read one row late (the segment of the next request leaks in)
    "ragged_rows_shifted": ("kv_rows_of", lambda kv, i: (int(kv[i]) + 1, int(kv[i + 1]) + 1)),
    # ragged K/V rows taken from the start of the tensor for every request
    "ragged_rows_from_zero": ("kv_rows_of", lambda kv, i: (0, int(kv[i + 1]) - int(kv[i]))),
    # drop the softmax scale
    "no_scale": ("attend", None),
    # transposed operand: V rows taken from K
    "v_from_k": ("attend", None),
    # log-sum-exp in log2 units where natural log is specified
    "lse_log2": ("attend", None),
}


def _mutated_attend(kind):
    import math

    def no_scale(q, K, V, lo, hi, scale):
        s = K[lo:hi + 1] @ q
        m = s.max()
        e = np.exp(s - m)
        return (e @ V[lo:hi + 1]) / e.sum(), m + math.log(e.sum())

    def v_from_k(q, K, V, lo, hi, scale):
        s = (K[lo:hi + 1] @ q) * scale
        m = s.max()
        e = np.exp(s - m)
        return (e @ K[lo:hi + 1]) / e.sum(), m + math.log(e.sum())

    def lse_log2(q, K, V, lo, hi, scale):
        s = (K[lo:hi + 1] @ q) * scale
        m = s.max()
        e = np.exp(s - m)
        return (e @ V[lo:hi + 1]) / e.sum(), m + math.log2(e.sum())

    return {"no_scale": no_scale, "v_from_k": v_from_k, "lse_log2": lse_log2}[kind]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(monkeypatch, name):
    attr, fn = MUTATIONS[name]
    if fn is None:
        fn = _mutated_attend(name)
    monkeypatch.setattr(A, attr, fn)
    assert not _all_pins_pass(), f"mutation {name} survived every pin"


def test_merge_with_swapped_weights_is_caught(monkeypatch):
    def bad(o1, s1, o2, s2):
        m = np.maximum(s1, s2)
        w1, w2 = np.exp(s2 - m), np.exp(s1 - m)
        return (o1 * w1 + o2 * w2) / (w1 + w2), m + np.log(w1 + w2)

    monkeypatch.setattr(A, "merge_states", bad)
    assert not P.check_merge_closed_form()


def test_csr_with_zero_remainder_is_caught(monkeypatch):
    # a remainder of 0 written as 0 instead of a full page
    monkeypatch.setattr(M, "last_page_len_for", lambda L, ps: L % ps)
    with pytest.raises(AssertionError):
        P.test_vllm_worked_example_slot_mapping_and_csr()


def test_merge_with_base2_weights_is_caught(monkeypatch):
    def bad(o1, s1, o2, s2):
        m = np.maximum(s1, s2)
        w1, w2 = np.exp2(s1 - m), np.exp2(s2 - m)  # natural-log LSEs weighted as if they were log2
        return (o1 * w1 + o2 * w2) / (w1 + w2), m + np.log(w1 + w2)

    monkeypatch.setattr(A, "merge_states", bad)
    assert not P.check_merge_closed_form()


def test_kv_store_with_page_and_offset_swapped_is_caught(monkeypatch):
    monkeypatch.setattr(A, "page_and_offset", lambda slot, ps: (slot % ps, slot // ps))
    with pytest.raises((AssertionError, IndexError)):
        P.test_kv_store_scatter_and_padding()


def _encode_ties_away(x):
    """E4M3 rounding to nearest with ties away from zero (a plausible wrong rounding mode)."""
    pos = F.decode_table()[:0x7F]  # codes 0x00..0x7E: the finite non-negative values, increasing
    xs = np.atleast_1d(np.asarray(x, dtype=np.float64))
    out = np.empty(xs.shape, dtype=np.uint8)
    for i, xi in enumerate(xs.ravel()):
        a = min(abs(xi), 448.0) if not np.isnan(xi) else 0.0
        j = int(np.searchsorted(pos, a))
        if j == 0:
            c = 0
        elif j >= len(pos):
            c = len(pos) - 1
        else:
            c = j if (a - pos[j - 1]) >= (pos[j] - a) else j - 1
        out.ravel()[i] = c | (0x80 if np.signbit(xi) else 0)
    return out if np.ndim(x) else out[0]


def test_fp8_ties_away_from_zero_is_caught(monkeypatch):
    monkeypatch.setattr(F, "encode", _encode_ties_away)
    with pytest.raises(AssertionError):
        P.test_e4m3_ties_round_to_even_and_saturate()


def test_fp8_without_saturation_is_caught(monkeypatch):
    orig = F.encode

    def no_sat(x):
        a = np.abs(np.asarray(x, dtype=np.float64))
        return np.where(a > 448.0, np.uint8(0x7F), orig(x)).astype(np.uint8)

    monkeypatch.setattr(F, "encode", no_sat)
    with pytest.raises(AssertionError):
        P.test_e4m3_ties_round_to_even_and_saturate()


def test_fp8_store_product_in_float64_is_caught(monkeypatch):
    monkeypatch.setattr(F, "quantize", lambda x, scale: F.encode(np.asarray(x, dtype=np.float64) / float(scale)))
    with pytest.raises(AssertionError):
        P.test_quantize_rounds_the_product_in_float32()



# ---- the plan metadata (slot mapping, CSR, page tables, decode-first split): worked-example pins ----
METADATA_MUTATIONS = {
    # offset taken from the logical page number and vice versa
    "slot_page_offset_swapped": ("slot_of", lambda row, pos, ps: int(row[pos % ps]) * ps + pos // ps),
    # the new tokens are the FIRST n positions of a request instead of the last n
    "new_tokens_first": ("slot_mapping", lambda bt, qsl, seq, ps: np.asarray(
        [M.slot_of(bt[i], p, ps) for i in range(len(seq)) for p in range(int(qsl[i + 1] - qsl[i]))], dtype=np.int64)),
    # page count rounded down
    "pages_floor": ("num_pages_for", lambda L, ps: L // ps),
    # the decode slice takes query length < threshold instead of <= threshold
    "decode_split_strict": ("decode_first_split", None),
    # token table sampled without the division by the page size
    "page_table_no_divide": ("page_table_from_token_table", lambda tt, seq, ps: np.stack(
        [np.asarray(tt[i][: int(max(seq)): ps]) for i in range(len(seq))]).astype(np.int64)),
    # page-size-1 view gathers every token from the first page of its request
    "ps1_view_page_blind": ("to_page_size_one", None),
}


def _strict_split(query_start_loc, threshold=1):
    qlen = np.diff(np.asarray(query_start_loc, dtype=np.int64))
    nd = int(np.sum(qlen < threshold))
    pq = np.concatenate([[0], np.cumsum(qlen[nd:])])
    return nd, int(qlen[:nd].sum()), len(qlen) - nd, int(qlen[nd:].sum()), pq


def _page_blind_ps1(kv_indptr, kv_indices, last_page_len, page_size):
    lens = M.kv_lens_from_csr(kv_indptr, last_page_len, page_size)
    slots, indptr = [], np.zeros(len(lens) + 1, dtype=np.int64)
    for i, L in enumerate(lens):
        first = int(kv_indices[kv_indptr[i]])
        slots += [first * page_size + j for j in range(int(L))]
        indptr[i + 1] = indptr[i] + int(L)
    return indptr, np.asarray(slots, dtype=np.int64), np.ones(len(lens), dtype=np.int64)


METADATA_PINS = [P.test_vllm_worked_example_slot_mapping_and_csr, P.test_minisgl_printed_metadata,
                 P.test_last_page_len_full_page_is_page_size_not_zero, P.test_to_page_size_one_matches_slot_formula]


@pytest.mark.parametrize("name", sorted(METADATA_MUTATIONS))
def test_metadata_pins_catch_planted_mistake(monkeypatch, name):
    attr, fn = METADATA_MUTATIONS[name]
    if fn is None:
        fn = {"decode_split_strict": _strict_split, "ps1_view_page_blind": _page_blind_ps1}[name]
    monkeypatch.setattr(M, attr, fn)
    failed = 0
    for pin in METADATA_PINS:
        try:
            pin()
        except (AssertionError, IndexError, ValueError):
            failed += 1
    assert failed > 0, f"mutation {name} survived every metadata pin"
