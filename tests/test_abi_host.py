"""The C ABI on the host (no GPU): every declared symbol is exported, the host helpers reproduce the
pages' worked examples, the planner rejects invalid batches loudly, and its split-KV / tile
partition covers every key of every (request, KV head) exactly once."""

import json
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def pk():
    from paged_kv_attention_slot_gb300 import build as B

    B.build()
    import paged_kv_attention_slot_gb300 as pk

    pk._lib.lib()
    return pk


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "pkv_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(pk):
    names = _declared_functions()
    assert len(names) >= 12
    L = pk._lib.lib()
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    assert sorted(names) == sorted(pk._lib.exported_symbols())


def test_block_table_to_csr_reproduces_worked_example(pk):
    g = json.load(open(os.path.join(GOLDEN, "vllm_worked_example.json")))
    indptr, indices, last = pk.block_table_to_csr(g["block_table"], g["seq_lens"], g["page_size"])
    e = g["expect"]
    assert indptr.tolist() == e["paged_kv_indptr"]
    assert indices.tolist() == e["paged_kv_indices"]
    assert last.tolist() == e["paged_kv_last_page_len"]


def test_token_table_to_page_table_reproduces_printed_example(pk):
    g = json.load(open(os.path.join(GOLDEN, "minisgl_metadata_example.json")))
    pt = pk.token_table_to_page_table(g["token_table"], g["device_len"], 4)
    assert pt.tolist() == g["expect"]["page_size_4"]["page_table"]
    # page size 1: the token table itself
    indptr, indices, last = pk.block_table_to_csr(g["token_table"], g["device_len"], 1)
    assert indptr.tolist() == g["expect"]["kv_indptr"]
    assert indices.tolist() == g["expect"]["kv_indices"]
    assert last.tolist() == g["expect"]["last_page_len"]


def _base(**kw):
    a = dict(qo_indptr=[0, 1, 2], kv_indptr=[0, 2, 3], kv_indices=[3, 1, 0], last_page_len=[5, 16],
             num_qo_heads=8, num_kv_heads=2, head_dim=128, page_size=16, mode="decode", num_sms=152)
    a.update(kw)
    return a


def _plan(pk, **kw):
    a = _base(**kw)
    idx = [a.pop(k) for k in ("qo_indptr", "kv_indptr", "kv_indices", "last_page_len")]
    return pk.Plan().plan(*idx, host_only=True, **a)


@pytest.mark.parametrize("bad, status", [
    (dict(qo_indptr=[1, 2, 3]), "PKV_EINVAL"),
    (dict(qo_indptr=[0, 2, 1]), "PKV_EINVAL"),
    (dict(kv_indptr=[1, 2, 3]), "PKV_EINVAL"),
    (dict(kv_indptr=[0, 3, 2]), "PKV_EINVAL"),
    (dict(last_page_len=[0, 16]), "PKV_EINVAL"),
    (dict(last_page_len=[17, 16]), "PKV_EINVAL"),
    (dict(kv_indices=[3, -1, 0]), "PKV_EINVAL"),
    (dict(num_qo_heads=6, num_kv_heads=4), "PKV_EINVAL"),
    (dict(head_dim=96), "PKV_EUNSUPPORTED"),
    (dict(qo_indptr=[0, 2, 3]), "PKV_EINVAL"),  # decode mode with two tokens in one request
    (dict(window_left=-2), "PKV_EINVAL"),
    (dict(page_size=0), "PKV_EINVAL"),
    (dict(kv_indptr=[0, 0, 1], kv_indices=[0], last_page_len=[0, 5]), "PKV_EINVAL"),  # a query but no keys
])
def test_plan_rejects_invalid_batches(pk, bad, status):
    with pytest.raises(pk.PkvError) as ei:
        _plan(pk, **bad)
    assert ei.value.args[0].startswith(status)


def test_run_on_host_only_plan_fails_loudly(pk):
    import ctypes as C

    p = _plan(pk)
    cache = pk._lib.pkv_cache(16, 16, 4, 16, 2, 128, 0, 4096, 256, 128, 1.0, 1.0)
    st = pk._lib.lib().pkv_attn_decode_run(p._h, 16, C.byref(cache), 16, None, None)
    assert st == pk._lib.PKV_EINVAL
    assert "host-only" in pk._lib.lib().pkv_last_error().decode()


@pytest.mark.parametrize("strides", [(0, 256, 128), (4096, 0, 128), (4096, 256, 0), (-4096, 256, 128),
                                     (4096, -256, 128), (4096, 256, -128)])
def test_noalloc_decode_rejects_non_positive_strides_before_any_launch(pk, strides):
    # the no-allocation decode runs the same cache checks as pkv_attn_decode_run: a zero or negative
    # stride (which passes the 16-byte test) would make the kernel gather outside the pool
    import ctypes as C

    p = _plan(pk)
    cache = pk._lib.pkv_cache(16, 16, 4, 16, 2, 128, 0, *strides, 1.0, 1.0)
    st = pk._lib.lib().pkv_attn_decode_run_noalloc(p._h, 16, C.byref(cache), 16, None, None)
    assert st == pk._lib.PKV_EINVAL
    assert "positive" in pk._lib.lib().pkv_last_error().decode()


def test_noalloc_decode_checks_the_cache_against_the_plan(pk):
    import ctypes as C

    p = _plan(pk)
    L = pk._lib.lib()
    for args in [(16, 16, 4, 16, 4, 128, 0, 4096, 256, 128, 1.0, 1.0),   # kv heads differ from the plan
                 (16, 16, 3, 16, 2, 128, 0, 4096, 256, 128, 1.0, 1.0),   # page 3 is beyond a 3-page pool
                 (24, 16, 4, 16, 2, 128, 0, 4096, 256, 128, 1.0, 1.0),   # misaligned pool pointer
                 (16, 16, 4, 16, 2, 128, 0, 4100, 256, 128, 1.0, 1.0)]:  # stride not a multiple of 16 B
        cache = pk._lib.pkv_cache(*args)
        assert L.pkv_attn_decode_run_noalloc(p._h, 16, C.byref(cache), 16, None, None) == pk._lib.PKV_EINVAL
    fp8 = _plan(pk, kv_dtype="e4m3")
    cache = pk._lib.pkv_cache(16, 16, 4, 16, 2, 128, 1, 4096, 256, 128, 0.0, 1.0)  # FP8 scale 0
    assert L.pkv_attn_decode_run_noalloc(fp8._h, 16, C.byref(cache), 16, None, None) == pk._lib.PKV_EINVAL
    assert "scale" in L.pkv_last_error().decode()


def _check_decode_cover(b, items, window=-1, group=None):
    """Every (request, kv head, head group) has its whole visible key range [lo, L) planned exactly once:
    either one CTA reading it alone (no partial slot), or several CTAs that share it (they claim its
    32-key groups at run time) with consecutive partial slots."""
    G = group
    groups = (G + 15) // 16
    seen = {}
    for req, h, hg, k0, k1, q_row, slot, q_rows in items.tolist():
        assert k0 < k1 and q_rows == 1
        seen.setdefault((req, h, hg), []).append((k0, k1, slot))
    for i, L in enumerate(b.kv_len.tolist()):
        lo = max(0, L - 1 - window) if window >= 0 else 0
        for h in range(b.num_kv_heads):
            for hg in range(groups):
                ranges = seen.pop((i, h, hg))
                assert all((k0, k1) == (lo, L) for k0, k1, _ in ranges)
                if len(ranges) == 1:
                    assert ranges[0][2] == -1
                else:
                    slots = sorted(r[2] for r in ranges)
                    assert slots == list(range(slots[0], slots[0] + len(slots)))
    assert not seen


@pytest.mark.parametrize("n", [2, 4])
def test_decode_partition_covers_every_key_once(pk, n):
    import workloads as W

    b = W.workload(n, scale_batch=0.25)
    p = pk.Plan().plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, num_qo_heads=b.num_qo_heads,
                       num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, page_size=b.page_size, mode="decode",
                       num_sms=152, host_only=True)
    items = p.work_items()
    info = p.info()
    _check_decode_cover(b, items, group=b.num_qo_heads // b.num_kv_heads)
    # longest first by the keys each CTA is expected to read (its range over the CTAs sharing it),
    # exact up to one bucket of the planner's counting sort: 2^s keys, the smallest s that puts the
    # longest share below B buckets, B = the number of CTAs clamped to [64, 4096]
    sharers = {}
    for r in items.tolist():
        sharers[(r[0], r[1], r[2])] = sharers.get((r[0], r[1], r[2]), 0) + 1
    ns = np.array([sharers[(r[0], r[1], r[2])] for r in items.tolist()])
    lens = (items[:, 4] - items[:, 3] + ns - 1) // ns
    buckets = min(4096, max(64, len(lens)))
    shift = 0
    while (int(lens.max()) >> shift) >= buckets:
        shift += 1
    assert np.all(np.diff(lens) < (1 << shift))
    assert info["kv_chunk"] % 64 == 0
    assert info["num_partials"] == int((items[:, 6] >= 0).sum())
    assert info["kv_tokens"] == int(b.kv_len.sum())


def test_decode_split_units_spread_over_the_launch_order(pk):
    # two 131,072-key FP8 requests x 8 KV heads: 16 split units of 38 CTAs each.  Equal shares are
    # launched split-major (split 0 of every unit, then split 1, ...), so every unit has CTAs in each
    # quarter of the launch order (the SMs' resident slots fill in launch order).
    import workloads as W

    b = W.workload(5)
    p = pk.Plan().plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, num_qo_heads=b.num_qo_heads,
                       num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, page_size=b.page_size, mode="decode",
                       kv_dtype="e4m3", num_sms=152, host_only=True)
    items = p.work_items()
    n = len(items)
    unit = items[:, 0] * b.num_kv_heads + items[:, 1]
    units = np.unique(unit)
    assert len(units) == 16 and n == 16 * (n // 16) and n // 16 > 8
    for u in units:
        pos = np.nonzero(unit == u)[0]
        quarters = np.bincount(pos * 4 // n, minlength=4)
        assert quarters.min() >= len(pos) // 4 - 1
    # round robin over the units: each run of 16 consecutive CTAs holds one CTA of every unit
    assert all(len(set(unit[i:i + 16].tolist())) == 16 for i in range(0, n, 16))
    _check_decode_cover(b, items, group=b.num_qo_heads // b.num_kv_heads)


def test_decode_order_with_more_ctas_than_buckets(pk):
    # 1,200 requests x 8 KV heads = 9,600 CTAs: the counting sort's bucket count is clamped at 4096
    rng = np.random.default_rng(17)
    B, ps = 1200, 16
    L = rng.integers(1, 5000, B)
    pages = (L + ps - 1) // ps
    kv_indptr = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
    idx = rng.permutation(int(kv_indptr[-1])).astype(np.int32)
    last = (L - (pages - 1) * ps).astype(np.int32)
    p = pk.Plan().plan(np.arange(B + 1, dtype=np.int32), kv_indptr, idx, last, num_qo_heads=32, num_kv_heads=8,
                       head_dim=128, page_size=ps, mode="decode", num_sms=152, host_only=True)
    items = p.work_items()
    assert len(items) > 4096
    sharers = {}
    for r in items.tolist():
        sharers[(r[0], r[1], r[2])] = sharers.get((r[0], r[1], r[2]), 0) + 1
    ns = np.array([sharers[(r[0], r[1], r[2])] for r in items.tolist()])
    lens = (items[:, 4] - items[:, 3] + ns - 1) // ns
    shift = 0
    while (int(lens.max()) >> shift) >= 4096:
        shift += 1
    assert np.all(np.diff(lens) < (1 << shift))
    # every key of every (request, KV head) is read by the CTAs of its unit
    for (req, h, g), n in list(sharers.items())[:50]:
        rows = items[(items[:, 0] == req) & (items[:, 1] == h)]
        assert rows[:, 3].min() == 0 and rows[:, 4].max() == L[req]


def test_window_partition_and_no_split(pk):
    import workloads as W

    b = W.make_batch([5000, 70, 4097], [1, 1, 1], 128, 32, 8, 128, seed=1, kv_dtype="e4m3")
    for w in (4096, 10):
        p = pk.Plan().plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, num_qo_heads=32, num_kv_heads=8,
                           head_dim=128, page_size=128, mode="decode", window_left=w, kv_dtype="e4m3",
                           num_sms=152, host_only=True)
        _check_decode_cover(b, p.work_items(), window=w, group=4)
    p = pk.Plan().plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, num_qo_heads=32, num_kv_heads=8,
                       head_dim=128, page_size=128, mode="decode", max_splits=1, kv_dtype="e4m3", num_sms=152,
                       host_only=True)
    assert p.info()["num_merge"] == 0 and len(p.work_items()) == 3 * 8


def test_large_group_uses_head_groups(pk):
    import workloads as W

    b = W.make_batch([300, 20], [1, 1], 16, 64, 2, 64, seed=2)
    p = pk.Plan().plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, num_qo_heads=64, num_kv_heads=2,
                       head_dim=64, page_size=16, mode="decode", num_sms=152, host_only=True)
    _check_decode_cover(b, p.work_items(), group=32)


def test_workspace_size_matches_plan(pk):
    a = _base()
    idx = [a.pop(k) for k in ("qo_indptr", "kv_indptr", "kv_indices", "last_page_len")]
    n = pk.Plan.workspace_size(*idx, **a)
    p = pk.Plan().plan(*idx, host_only=True, **a)
    assert p.info()["workspace_bytes"] == n and n % 256 == 0


def _mixed_plan(pk, order):
    """The worked example's three requests (A decode, B 4-token prefill, C 3-token extend) in `order`."""
    g = json.load(open(os.path.join(GOLDEN, "vllm_worked_example.json")))
    q_lens = np.diff(g["query_start_loc"]).tolist()
    rows = [g["block_table"][i] for i in order]
    seq = [g["seq_lens"][i] for i in order]
    ql = [q_lens[i] for i in order]
    indptr, indices, last = pk.block_table_to_csr(rows, seq, g["page_size"])
    qo = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    p = pk.Plan().plan(qo, indptr, indices, last, num_qo_heads=32, num_kv_heads=8, head_dim=128,
                       page_size=g["page_size"], mode="mixed", num_sms=152, host_only=True)
    return g, p, qo


@pytest.mark.parametrize("order", [[0, 1, 2], [1, 0, 2], [2, 1, 0]])
def test_mixed_plan_splits_decode_and_extend_as_printed(pk, order):
    """Mixed batch: the decode/extend counts and the extend slice's query offsets are the printed ones,
    whatever the request order (each CTA carries its own token row, so no decode-first reorder)."""
    g, p, qo = _mixed_plan(pk, order)
    e = g["expect"]
    info = p.info()
    assert info["mode"] == pk._lib.PKV_MODE_MIXED
    for k in ("num_decodes", "num_decode_tokens", "num_prefills", "num_prefill_tokens"):
        assert info[k] == e[k]
    items = p.work_items()
    nd = info["num_decode_work"]
    dec, pre = items[:nd], items[nd:]
    a_pos = order.index(0)  # request A is the decode request
    assert set(dec[:, 0].tolist()) == {a_pos} and set(dec[:, 5].tolist()) == {int(qo[a_pos])}
    assert len(dec) == 8  # one CTA per KV head: 128 keys are one chunk
    assert a_pos not in set(pre[:, 0].tolist())
    # per KV head, the extend CTAs cover B's and C's rows; in the printed order their query counts
    # give the prefill slice's qo_indptr
    for h in range(8):
        mine = pre[pre[:, 1] == h]
        got = {int(r[0]): (int(r[5]), int(r[7])) for r in mine}
        want = {i: (int(qo[i]), int(qo[i + 1] - qo[i])) for i in range(3) if i != a_pos}
        assert got == want
    if order == [0, 1, 2]:
        q_rows = [int(r[7]) for r in sorted(pre[pre[:, 1] == 0].tolist(), key=lambda r: r[5])]
        assert np.concatenate([[0], np.cumsum(q_rows)]).tolist() == e["prefill_qo_indptr"]


def test_mixed_plan_with_only_decodes_needs_no_prefill_support(pk):
    """A mixed plan whose requests all have one new token is a decode plan (FP8 KV allowed)."""
    p = pk.Plan().plan([0, 1, 2], [0, 2, 3], [3, 1, 0], [5, 16], num_qo_heads=32, num_kv_heads=8, head_dim=128,
                       page_size=16, mode="mixed", kv_dtype="e4m3", num_sms=152, host_only=True)
    info = p.info()
    assert info["num_decode_work"] == info["num_work"] == 2 * 8 and info["num_prefills"] == 0
    with pytest.raises(pk.PkvError):  # an extend request with an FP8 cache is not supported
        pk.Plan().plan([0, 1, 3], [0, 2, 3], [3, 1, 0], [5, 16], num_qo_heads=32, num_kv_heads=8, head_dim=128,
                       page_size=16, mode="mixed", kv_dtype="e4m3", num_sms=152, host_only=True)


# ---- ragged (contiguous K/V) and non-causal plans -------------------------------------------------
def _extend(**kw):
    a = dict(qo_indptr=[0, 40, 41, 300], kv_indptr=[0, 2, 3, 20], kv_indices=list(range(20)),
             last_page_len=[10, 16, 16], num_qo_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
             mode="prefill", num_sms=152)
    a.update(kw)
    idx = [a.pop(k) for k in ("qo_indptr", "kv_indptr", "kv_indices", "last_page_len")]
    return pk_plan_host(*idx, **a)


def pk_plan_host(*idx, **a):
    import paged_kv_attention_slot_gb300 as pk

    return pk.Plan().plan(*idx, host_only=True, **a)


@pytest.mark.parametrize("bad, status", [
    (dict(causal=False, mode="decode", qo_indptr=[0, 1, 2, 3]), "PKV_EINVAL"),  # non-causal decode plan
    (dict(causal=False, mode="mixed"), "PKV_EINVAL"),
    (dict(causal=False, window_left=16), "PKV_EINVAL"),  # a window needs the causal mask
    (dict(mode="ragged", kv_indptr=[0, 50, 40, 300]), "PKV_EINVAL"),  # ragged rows not non-decreasing
    (dict(mode="ragged", kv_indptr=[0, 39, 40, 300]), "PKV_EINVAL"),  # causal: 39 keys for 40 queries
    (dict(mode="ragged", kv_indptr=[1, 40, 41, 300]), "PKV_EINVAL"),
])
def test_plan_rejects_invalid_ragged_and_noncausal(pk, bad, status):
    with pytest.raises(pk.PkvError) as ei:
        _extend(**bad)
    assert ei.value.args[0].startswith(status)


def test_status_codes_of_causal_argument(pk):
    import ctypes as C

    a, keep = pk.Plan._args([0, 2], [0, 1], [0], [2], 8, 2, 128, 16, "prefill", -1, 0.0, "bf16", 0, 152)
    a.causal = 2
    n = C.c_size_t(0)
    assert pk._lib.lib().pkv_plan_workspace_size(C.byref(a), C.byref(n)) == pk._lib.PKV_EINVAL


def _prefill_items(p):
    return [tuple(r) for r in p.work_items()[p.info()["num_decode_work"]:].tolist()]


def test_ragged_plan_reads_each_requests_rows(pk):
    # self-attention over fresh segments: kv rows = qo rows, causal, no page table at all
    qo = [0, 5, 5, 300, 301]
    p = pk.Plan().plan(qo, qo, None, None, num_qo_heads=8, num_kv_heads=2, head_dim=128, mode="ragged",
                       num_sms=152, host_only=True)
    info = p.info()
    assert info["max_page_id"] == 300  # the largest K/V row read
    assert info["num_prefill_tokens"] == 301
    tok = 2 * 128 // 4  # tokens per CTA (two 128-row tiles of 4 heads per KV head)
    for req, h, hg, k0, k1, q_row, slot, q_rows in _prefill_items(p):
        n = qo[req + 1] - qo[req]
        t0 = q_row - qo[req]
        assert k0 == 0 and k1 == min(t0 + tok, n) and q_rows == min(tok, n - t0)  # causal: keys up to the last row


def test_noncausal_plan_reads_the_whole_segment_and_allows_short_or_empty_ones(pk):
    # the prefix pass of an extend: L_i prefix keys, n_i > L_i allowed, L_i = 0 gives an empty item
    qo = [0, 100, 130, 200]
    kv_len = [7, 0, 1000]
    ps = 16
    pages = [(L + ps - 1) // ps for L in kv_len]
    indptr = np.concatenate([[0], np.cumsum(pages)]).tolist()
    last = [L - (n - 1) * ps if n else 0 for L, n in zip(kv_len, pages)]
    p = pk.Plan().plan(qo, indptr, list(range(indptr[-1])), last, num_qo_heads=8, num_kv_heads=2, head_dim=128,
                       page_size=ps, mode="prefill", causal=False, num_sms=152, max_splits=1, host_only=True)
    for req, h, hg, k0, k1, q_row, slot, q_rows in _prefill_items(p):
        assert (k0, k1) == (0, kv_len[req])
    # with splitting allowed, the pieces of each (request, head, query tile) still cover [0, L) once
    p = pk.Plan().plan(qo, indptr, list(range(indptr[-1])), last, num_qo_heads=8, num_kv_heads=2, head_dim=128,
                       page_size=ps, mode="prefill", causal=False, num_sms=152, host_only=True)
    cover = {}
    for req, h, hg, k0, k1, q_row, slot, q_rows in _prefill_items(p):
        cover.setdefault((req, h, q_row), []).append((k0, k1))
    for (req, h, q_row), pieces in cover.items():
        pieces.sort()
        assert pieces[0][0] == 0 and pieces[-1][1] == kv_len[req]
        assert all(a[1] == b_[0] for a, b_ in zip(pieces, pieces[1:]))


def test_merge_state_argument_checks(pk):
    L = pk._lib.lib()
    assert L.pkv_merge_state(None, None, None, None, None, None, 0, 128, None) == pk._lib.PKV_OK  # no states
    assert L.pkv_merge_state(16, 16, 16, 16, 16, None, 4, 96, None) == pk._lib.PKV_EUNSUPPORTED
    assert L.pkv_merge_state(16, 16, None, 16, 16, None, 4, 128, None) == pk._lib.PKV_EINVAL
    assert L.pkv_merge_state(16, 16, 16, 16, 16, None, -1, 128, None) == pk._lib.PKV_EINVAL


# ---- prefill split-KV --------------------------------------------------------------------------------
def _prefill_pieces(p):
    info = p.info()
    return p.work_items()[info["num_decode_work"]:], info


@pytest.mark.parametrize("causal, window", [(True, -1), (False, -1), (True, 3000)])
def test_prefill_split_covers_every_key_once(pk, causal, window):
    # few items (one request, 2 KV heads, 64 tokens): long key ranges are cut into 128-key-tile chunks
    L, n, ps = 20000, 64, 16
    npg = (L + ps - 1) // ps
    p = pk.Plan().plan([0, n], [0, npg], list(range(npg)), [L - (npg - 1) * ps], num_qo_heads=8, num_kv_heads=2,
                       head_dim=128, page_size=ps, mode="prefill", causal=causal, window_left=window,
                       num_sms=152, host_only=True)
    items, info = _prefill_pieces(p)
    assert info["num_prefill_partials"] == len(items) > 2
    by_head = {}
    for req, h, hg, k0, k1, q_row, slot, q_rows in items.tolist():
        assert slot >= 0 and q_rows == n and q_row == 0
        by_head.setdefault(h, []).append((k0, k1, slot))
    lo = 0 if window < 0 else max(0, L - n - window)
    hi = L if not causal else L  # causal: the last row is at position L - 1
    slots = []
    for h, pieces in by_head.items():
        pieces.sort()
        assert pieces[0][0] == lo and pieces[-1][1] == hi
        for (a0, a1, _), (b0, b1, _) in zip(pieces, pieces[1:]):
            assert a1 == b0 and (a1 - a0) % 128 == 0
        slots += [s_ for _, _, s_ in pieces]
    assert sorted(slots) == list(range(len(slots)))
    assert info["num_merge"] == 2


def test_prefill_split_respects_max_splits_and_many_items(pk):
    L, n, ps = 20000, 64, 16
    npg = (L + ps - 1) // ps
    args = ([0, n], [0, npg], list(range(npg)), [L - (npg - 1) * ps])
    kw = dict(num_qo_heads=8, num_kv_heads=2, head_dim=128, page_size=ps, mode="prefill", host_only=True)
    never = pk.Plan().plan(*args, max_splits=1, num_sms=152, **kw)
    assert never.info()["num_prefill_partials"] == 0 and never.info()["num_work"] == 2
    three = pk.Plan().plan(*args, max_splits=3, num_sms=152, **kw)
    assert three.info()["num_work"] == 6 and three.info()["num_prefill_partials"] == 6
    # the prefix-extend workload fills many waves on its own: no split
    import workloads as W

    b = W.workload(3)
    big = pk.Plan().plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, num_qo_heads=32, num_kv_heads=8,
                         head_dim=128, page_size=1, mode="prefill", num_sms=152, host_only=True)
    assert big.info()["num_prefill_partials"] == 0 and big.info()["num_merge"] == 0


def test_prefill_run_merge_argument_checks(pk):
    import ctypes as C

    L = pk._lib.lib()
    # a host-only plan cannot run; a decode plan cannot merge; a merging run needs the held lse
    p = pk.Plan().plan([0, 40], [0, 3], [0, 1, 2], [16], num_qo_heads=8, num_kv_heads=2, head_dim=128,
                       page_size=16, mode="prefill", num_sms=152, host_only=True)
    cache = pk._lib.pkv_cache(16, 16, 4, 16, 2, 128, 0, 4096, 256, 128, 1.0, 1.0)
    assert L.pkv_attn_prefill_run_merge(p._h, 16, C.byref(cache), 16, None, None) == pk._lib.PKV_EINVAL
    assert L.pkv_attn_prefill_run_merge(None, 16, C.byref(cache), 16, 16, None) == pk._lib.PKV_EINVAL
    assert "plan" in L.pkv_last_error().decode()


def test_plan_from_read_only_and_non_int32_arrays(pk):
    # the binding reads array addresses through the buffer protocol, falling back for read-only
    # buffers; int64 / list inputs are converted: all of them must give the same plan
    import workloads as W

    b = W.workload(2, scale_batch=0.25)
    kw = dict(num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads, head_dim=b.head_dim,
              page_size=b.page_size, mode="decode", num_sms=152, host_only=True)
    ref = pk.Plan().plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, **kw).work_items()
    ro = [np.array(a, dtype=np.int32) for a in (b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len)]
    for a in ro:
        a.flags.writeable = False
    got_ro = pk.Plan().plan(*ro, **kw).work_items()
    got_64 = pk.Plan().plan(*[np.asarray(a, dtype=np.int64) for a in ro], **kw).work_items()
    got_list = pk.Plan().plan(*[a.tolist() for a in ro], **kw).work_items()
    for got in (got_ro, got_64, got_list):
        assert np.array_equal(got, ref)


def _random_batch(rng, mode):
    """A random CSR batch for the planner fuzz test: lengths, pages, a random page permutation."""
    B = int(rng.integers(1, 25))
    ps = int(rng.choice([1, 4, 16, 64]))
    if mode == "decode":
        n = rng.choice([0, 1, 1, 1], B)
    elif mode == "prefill":
        n = rng.integers(1, 300, B)
    else:
        n = np.where(rng.random(B) < 0.5, 1, rng.integers(2, 300, B))
    L = n + rng.integers(0, 700, B)
    L = np.where((n == 0) & (rng.random(B) < 0.3), 0, L)
    pages = (L + ps - 1) // ps
    kv_indptr = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
    idx = rng.permutation(int(kv_indptr[-1]) + 5)[: int(kv_indptr[-1])].astype(np.int32)
    last = np.where(pages > 0, L - (pages - 1) * ps, 1).astype(np.int32)
    qo = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    return qo, kv_indptr, idx, last, ps, n.astype(np.int64), L.astype(np.int64)


@pytest.mark.parametrize("seed", range(60))
def test_planner_fuzz_partitions(pk, seed):
    """Random batches, modes, head ratios, windows, SM counts and split caps: every visible key range
    is planned exactly once (decode units: one CTA or CTAs sharing the range with consecutive slots;
    prefill items: pieces that tile the item's range with consecutive slots) and every new token row
    is covered exactly once."""
    rng = np.random.default_rng(9000 + seed)
    mode = ["decode", "prefill", "mixed"][seed % 3]
    qo, kv_indptr, idx, last, ps, n, L = _random_batch(rng, mode)
    hkv = int(rng.choice([1, 2, 8]))
    G = int(rng.choice([1, 4, 8, 16, 32]))
    window = -1 if rng.random() < 0.5 else int(rng.integers(0, 400))
    p = pk.Plan().plan(qo, kv_indptr, idx, last, num_qo_heads=hkv * G, num_kv_heads=hkv, head_dim=128,
                       page_size=ps, mode=mode, window_left=window, num_sms=int(rng.choice([8, 40, 152])),
                       max_splits=int(rng.choice([0, 1, 3])), host_only=True)
    info = p.info()
    items = p.work_items()
    nd = info["num_decode_work"]
    assert info["num_work"] == len(items)
    is_decode = (n == 1) if mode != "prefill" else np.zeros(len(n), dtype=bool)
    # decode units
    groups = (G + 15) // 16
    seen = {}
    for req, h, hg, k0, k1, q_row, slot, q_rows in items[:nd].tolist():
        assert is_decode[req] and q_rows == 1 and q_row == qo[req]
        seen.setdefault((req, h, hg), []).append((k0, k1, slot))
    for i in np.nonzero(is_decode)[0].tolist():
        lo = max(0, int(L[i]) - 1 - window) if window >= 0 else 0
        for h in range(hkv):
            for hg in range(groups):
                ranges = seen.pop((i, h, hg))
                assert all((k0, k1) == (lo, int(L[i])) for k0, k1, _ in ranges)
                slots = sorted(r[2] for r in ranges)
                assert slots == [-1] if len(ranges) == 1 else slots == list(range(slots[0], slots[0] + len(slots)))
    assert not seen
    # prefill items: group the pieces of each (request, KV head, first row)
    pieces = {}
    for req, h, hg, k0, k1, q_row, slot, q_rows in items[nd:].tolist():
        assert not is_decode[req] and n[req] > 0 and 0 < q_rows <= 2 * (128 // G)
        pieces.setdefault((req, h, q_row, q_rows), []).append((k0, k1, slot))
    rows = {}
    for (req, h, q_row, q_rows), rs in pieces.items():
        t0 = q_row - int(qo[req])
        P0 = int(L[req] - n[req]) + t0
        lo = max(0, P0 - window) if window >= 0 else 0
        hi = P0 + q_rows  # the last row's position + 1 (causal)
        rs.sort()
        assert rs[0][0] == lo and rs[-1][1] == hi
        assert all(a[1] == b[0] for a, b in zip(rs, rs[1:]))  # the pieces tile [lo, hi)
        slots = [r[2] for r in rs]
        assert slots == [-1] if len(rs) == 1 else slots == list(range(slots[0], slots[0] + len(slots)))
        rows.setdefault((req, h), []).append((q_row, q_rows))
    for i in np.nonzero((~is_decode) & (n > 0))[0].tolist():
        for h in range(hkv):
            spans = sorted(rows.pop((i, h)))
            assert spans[0][0] == qo[i] and sum(r for _, r in spans) == n[i]
            assert all(a[0] + a[1] == b[0] for a, b in zip(spans, spans[1:]))
    assert not rows



def test_binding_rejects_malformed_pools_and_kv_writes(pk):
    # the binding's own checks, raised before any call into the library (no GPU needed)
    import torch

    ok = torch.zeros((4, 16, 2, 128), dtype=torch.bfloat16)
    pk.KVCache(ok, ok.clone())  # well-formed
    pk.KVCache(ok.to(torch.uint8), ok.to(torch.uint8), 0.5, 0.25)  # FP8 codes with scales
    bad = [
        (ok[0], ok[0]),                                            # not 4-D
        (ok, ok[:, :8]),                                           # shapes differ
        (ok.transpose(2, 3), ok.transpose(2, 3)),                  # head_dim not contiguous
        (ok.float(), ok.float()),                                  # unsupported dtype
        (ok, ok.to(torch.uint8)),                                  # K and V dtypes differ
        (ok, torch.zeros((4, 2, 16, 128), dtype=torch.bfloat16).transpose(1, 2)),  # strides differ
    ]
    for k, v in bad:
        with pytest.raises(ValueError):
            pk.KVCache(k, v)
    cache = pk.KVCache(ok, ok.clone())
    k = torch.zeros((3, 2, 128), dtype=torch.bfloat16)
    slots = torch.zeros(3, dtype=torch.int64)
    for args in [
        (k.float(), k, slots),                                     # not bf16
        (k.transpose(0, 1).contiguous().transpose(0, 1), k, slots),  # not contiguous
        (k, k, slots.int()),                                       # slot_mapping not int64
        (k, k, slots[:2]),                                         # one slot per token
        (k[:, :1], k[:, :1], slots),                               # heads do not match the pool
    ]:
        with pytest.raises(ValueError):
            pk.kv_store(*args, cache)


@pytest.mark.parametrize("seed", range(8))
def test_host_helpers_match_the_oracle_on_random_tables(pk, seed):
    from oracle import metadata as M

    rng = np.random.default_rng(300 + seed)
    B = int(rng.integers(1, 12))
    ps = int(rng.choice([1, 2, 16, 64]))
    seq = rng.integers(0, 500, B)
    max_pages = int(max(1, ((seq + ps - 1) // ps).max()))
    bt = rng.integers(0, 10_000, (B, max_pages + int(rng.integers(0, 3)))).astype(np.int32)
    got = pk.block_table_to_csr(bt, seq, ps)
    want = M.csr_from_block_table(bt, seq, ps)
    assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1])
    has = (seq > 0)
    assert np.array_equal(np.asarray(got[2])[has], np.asarray(want[2])[has])  # a request of length 0 has no page
    if seq.max() > 0:
        tt = rng.integers(0, 1 << 20, (B, int(seq.max()) + int(rng.integers(0, 4)))).astype(np.int32)
        assert np.array_equal(pk.token_table_to_page_table(tt, seq, ps), M.page_table_from_token_table(tt, seq, ps))


def test_prefill_order_groups_requests_and_kv_heads_with_a_longest_first_tail(pk):
    # prefill CTAs come group by group ((request, KV head), largest total first, each group longest
    # first) so that the CTAs resident together share K/V rows in L2; the last ~10 % of the work is
    # longest first again, so no long item starts near the end.  Every key is still planned once.
    import workloads as W

    b = W.workload(3)
    p = pk.Plan().plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, num_qo_heads=32,
                       num_kv_heads=8, head_dim=128, page_size=1, mode="prefill", num_sms=152, host_only=True)
    it = p.work_items()  # req, kv_head, head_group, kv_begin, kv_end, q_row, out_slot, q_rows
    share = (it[:, 4] - it[:, 3]).astype(np.int64)
    total = share.sum()
    cut = int(np.searchsorted(np.cumsum(share), 0.9 * total, side="right")) + 1
    head, tail = it[:cut], share[cut:]
    # the tail is longest first (up to the counting sort's bucket width)
    assert np.all(np.diff(tail) <= share.max() // 64 + 1)
    # the head is a sequence of contiguous groups, largest group total first, each longest first
    groups = head[:, 0] * 8 + head[:, 1]
    starts = np.flatnonzero(np.r_[True, groups[1:] != groups[:-1]])
    assert len(starts) == len(np.unique(groups)), "a group is split in the head"
    g_total = {g: share[(it[:, 0] * 8 + it[:, 1]) == g].sum() for g in np.unique(groups)}
    seq = [g_total[groups[s0]] for s0 in starts]
    assert all(x >= y for x, y in zip(seq, seq[1:]))
    for s0, s1 in zip(starts, list(starts[1:]) + [cut]):
        assert np.all(np.diff(share[s0:s1]) <= share.max() // 64 + 1)


def test_paged_ragged_plan_spans_prefix_and_new_rows(pk):
    # PKV_MODE_PAGED_RAGGED: the page table holds only the prefix; each request's key range is its
    # prefix plus its new tokens, planned exactly as the single causal paged pass over both
    ps = 16
    pre, n = [0, 100, 4096, 33], [50, 1, 300, 0]
    npg = [(x + ps - 1) // ps for x in pre]
    indptr = np.concatenate([[0], np.cumsum(npg)]).astype(np.int32)
    indices = np.arange(indptr[-1], dtype=np.int32)
    last = np.array([x - (k - 1) * ps if k else 0 for x, k in zip(pre, npg)], np.int32)
    qo = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    kw = dict(num_qo_heads=8, num_kv_heads=2, head_dim=128, page_size=ps, num_sms=152, host_only=True)
    p = pk.Plan().plan(qo, indptr, indices, last, mode="paged_ragged", **kw)
    # the same batch as one paged pool holding prefix + new tokens
    full = [x + y for x, y in zip(pre, n)]
    fpg = [(x + ps - 1) // ps for x in full]
    findptr = np.concatenate([[0], np.cumsum(fpg)]).astype(np.int32)
    flast = np.array([x - (k - 1) * ps if k else 0 for x, k in zip(full, fpg)], np.int32)
    f = pk.Plan().plan(qo, findptr, np.arange(findptr[-1], dtype=np.int32), flast, mode="prefill", **kw)
    a, b = p.work_items(), f.work_items()
    # same CTAs (request, KV head, key range, rows); only the page-list base differs
    key = lambda it: sorted(map(tuple, it[:, [0, 1, 3, 4, 5, 7]].tolist()))
    assert key(a) == key(b)
    assert p.info()["kv_tokens"] == f.info()["kv_tokens"]
    assert p.info()["max_page_id"] == int(indices.max())
    # non-causal plans are allowed; decode-style checks do not apply
    pk.Plan().plan(qo, indptr, indices, last, mode="paged_ragged", causal=False, **kw)


def test_paged_ragged_argument_checks(pk):
    import ctypes as C

    L = pk._lib.lib()
    kw = dict(num_qo_heads=8, num_kv_heads=2, head_dim=128, page_size=16, num_sms=152, host_only=True)
    args = ([0, 40], [0, 3], [0, 1, 2], [16])
    p = pk.Plan().plan(*args, mode="paged_ragged", **kw)
    f = pk.Plan().plan(*args, mode="prefill", **kw)
    cache = pk._lib.pkv_cache(16, 16, 4, 16, 2, 128, 0, 4096, 256, 128, 1.0, 1.0)
    # a prefill plan cannot run as paged + ragged, nor a paged + ragged plan as prefill
    assert L.pkv_attn_paged_ragged_run(f._h, 16, C.byref(cache), 16, 16, 16, None, None) == pk._lib.PKV_EINVAL
    assert "PKV_MODE_PAGED_RAGGED" in L.pkv_last_error().decode()
    assert L.pkv_attn_prefill_run(p._h, 16, C.byref(cache), 16, None, None) == pk._lib.PKV_EINVAL
    # the new rows are required and must be 16-byte aligned
    assert L.pkv_attn_paged_ragged_run(p._h, 16, C.byref(cache), None, 16, 16, None, None) == pk._lib.PKV_EINVAL
    assert L.pkv_attn_paged_ragged_run(p._h, 16, C.byref(cache), 24, 16, 16, None, None) == pk._lib.PKV_EINVAL
    # the prefill kernel reads a bf16 cache only
    with pytest.raises(pk.PkvError) as ei:
        pk.Plan().plan(*args, mode="paged_ragged", kv_dtype="e4m3", **kw)
    assert ei.value.args[0].startswith("PKV_EUNSUPPORTED")


def test_cascade_run_argument_checks(pk):
    # pkv_cascade_run: a non-causal prefill plan over the shared pages for every query row, and a
    # suffix plan over the same rows; mismatches fail before anything is enqueued
    import ctypes as C

    L = pk._lib.lib()
    kw = dict(num_kv_heads=2, head_dim=128, page_size=16, num_sms=152, host_only=True)
    shared = pk.Plan().plan([0, 3], [0, 4], [0, 1, 2, 3], [16], num_qo_heads=8, mode="prefill", causal=False, **kw)
    causal_shared = pk.Plan().plan([0, 3], [0, 4], [0, 1, 2, 3], [16], num_qo_heads=8, mode="prefill", **kw)
    suffix = pk.Plan().plan([0, 1, 2, 3], [0, 1, 2, 3], [4, 5, 6], [3, 7, 16], num_qo_heads=8, mode="decode", **kw)
    other_heads = pk.Plan().plan([0, 1, 2, 3], [0, 1, 2, 3], [4, 5, 6], [3, 7, 16], num_qo_heads=16, mode="decode", **kw)
    two_rows = pk.Plan().plan([0, 1, 2], [0, 1, 2], [4, 5], [3, 7], num_qo_heads=8, mode="decode", **kw)
    cache = pk._lib.pkv_cache(16, 16, 8, 16, 2, 128, 0, 4096, 256, 128, 1.0, 1.0)
    run = lambda a, b, lse=16: L.pkv_cascade_run(a._h, b._h, 16, C.byref(cache), 16, lse, None)  # noqa: E731
    for a, b, msg in [(causal_shared, suffix, "non-causal"), (shared, other_heads, "same heads"),
                      (shared, two_rows, "same heads"), (suffix, suffix, "non-causal")]:
        assert run(a, b) == pk._lib.PKV_EINVAL
        assert msg in L.pkv_last_error().decode()
    assert run(shared, suffix, lse=None) == pk._lib.PKV_EINVAL
    assert "lse is required" in L.pkv_last_error().decode()
    assert run(shared, suffix) == pk._lib.PKV_EINVAL  # host-only plans cannot run
    assert "host-only" in L.pkv_last_error().decode()


def test_wait_limit_and_hold_settings(pk):
    # the bound on the prefill kernel's waits: <= 0 restores the default, beyond 2^41 clocks is
    # rejected; the hold switch only toggles (its effect is exercised on the GPU)
    L = pk._lib.lib()
    assert L.pkv_set_wait_limit(20000) == pk._lib.PKV_OK
    assert L.pkv_set_wait_limit(0) == pk._lib.PKV_OK
    assert L.pkv_set_wait_limit(-5) == pk._lib.PKV_OK
    assert L.pkv_set_wait_limit(1 << 42) == pk._lib.PKV_EINVAL
    assert "too large" in L.pkv_last_error().decode()
    assert L.pkv_test_hold_wait(1) == pk._lib.PKV_OK
    assert L.pkv_test_hold_wait(0) == pk._lib.PKV_OK
    pk.set_wait_limit(0)
