"""Pins of the CPU oracle against values and facts that do not come from the oracle itself.

Each check below is written independently of the oracle's helpers: the worked
examples printed on the pages (tests/golden/), brute force with Python loops,
the library routine the pages' own CPU reference calls
(torch.nn.functional.scaled_dot_product_attention with enable_gqa), closed
forms (single visible key, uniform scores, split-and-merge) and invariants the
pages state (page-size-1 view, physical page permutation).  test_oracle_mutations.py
plants plausible mistakes in the oracle and checks that these pins catch them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import fp8 as F
from oracle import metadata as M

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------------------------
# metadata: worked examples printed on the pages
# ---------------------------------------------------------------------------------------------
def test_vllm_worked_example_slot_mapping_and_csr():
    g = _golden("vllm_worked_example.json")
    ps = g["page_size"]
    e = g["expect"]
    sm = M.slot_mapping(g["block_table"], g["query_start_loc"], g["seq_lens"], ps)
    assert sm.tolist() == e["slot_mapping"]
    indptr, indices, last = M.csr_from_block_table(g["block_table"], g["seq_lens"], ps)
    assert indptr.tolist() == e["paged_kv_indptr"]
    assert indices.tolist() == e["paged_kv_indices"]
    assert last.tolist() == e["paged_kv_last_page_len"]
    nd, ndt, npf, npft, pq = M.decode_first_split(g["query_start_loc"])
    assert (nd, ndt, npf, npft) == (e["num_decodes"], e["num_decode_tokens"], e["num_prefills"], e["num_prefill_tokens"])
    assert pq.tolist() == e["prefill_qo_indptr"]
    assert max(np.diff(g["query_start_loc"])) == e["max_query_len"]
    assert max(g["seq_lens"]) == e["max_seq_len"]
    # the inverse encoding recovers the lengths
    assert M.kv_lens_from_csr(indptr, last, ps).tolist() == g["seq_lens"]


def test_minisgl_printed_metadata():
    g = _golden("minisgl_metadata_example.json")
    e = g["expect"]
    dev, cached = g["device_len"], g["cached_len"]
    qo = np.concatenate([[0], np.cumsum(np.subtract(dev, cached))])
    assert qo.tolist() == e["qo_indptr"]
    indptr, indices, last = M.token_csr_from_token_table(g["token_table"], dev)
    assert indptr.tolist() == e["kv_indptr"]
    assert indices.tolist() == e["kv_indices"]
    assert last.tolist() == e["last_page_len"]
    pt = M.page_table_from_token_table(g["token_table"], dev, 4)
    assert pt.tolist() == e["page_size_4"]["page_table"]
    assert list(dev) == e["page_size_4"]["cache_seqlens"]
    # page-size-1 slots of the new tokens (what the page's batch_of() writes to)
    sm = M.slot_mapping(g["token_table"], qo, dev, 1)
    assert sm.tolist() == e["out_loc"]


def test_last_page_len_full_page_is_page_size_not_zero():
    assert M.last_page_len_for(32, 16) == 16
    assert M.last_page_len_for(33, 16) == 1
    assert M.last_page_len_for(1, 16) == 1
    assert M.num_pages_for(32, 16) == 2
    assert M.num_pages_for(33, 16) == 3
    assert M.num_pages_for(0, 16) == 0


def test_to_page_size_one_matches_slot_formula():
    g = _golden("vllm_worked_example.json")
    ps = g["page_size"]
    indptr, indices, last = M.csr_from_block_table(g["block_table"], g["seq_lens"], ps)
    p1, s1, l1 = M.to_page_size_one(indptr, indices, last, ps)
    assert p1.tolist() == [0, 128, 132, 167]
    assert l1.tolist() == [1, 1, 1]
    # request A's position 127 is the worked example's slot 175; C's position 34 is slot 194
    assert s1[127] == 175 and s1[128 + 4 + 34] == 194


# ---------------------------------------------------------------------------------------------
# FP8 E4M3 codec
# ---------------------------------------------------------------------------------------------
def test_e4m3_known_codes():
    d = F.decode_table()
    assert d[0x00] == 0.0 and not np.signbit(d[0x00])
    assert d[0x80] == 0.0 and np.signbit(d[0x80])
    assert d[0x01] == 2.0 ** -9
    assert d[0x07] == 7 * 2.0 ** -9
    assert d[0x08] == 2.0 ** -6
    assert d[0x38] == 1.0
    assert d[0x3C] == 1.5
    assert d[0x7E] == 448.0
    assert d[0xFE] == -448.0
    assert np.isnan(d[0x7F]) and np.isnan(d[0xFF])
    assert np.sum(np.isnan(d)) == 2


def test_e4m3_roundtrip_every_finite_code():
    d = F.decode_table()
    codes = np.array([c for c in range(256) if not np.isnan(d[c])])
    assert np.array_equal(F.encode(d[codes]), codes.astype(np.uint8))


def test_e4m3_ties_round_to_even_and_saturate():
    d = F.decode_table()
    pos = [c for c in range(0x00, 0x7E)]  # consecutive finite positive codes c, c+1
    for c in pos:
        mid = (d[c] + d[c + 1]) / 2.0
        want = c if c % 2 == 0 else c + 1  # the even mantissa wins the tie
        assert F.encode(mid) == want, hex(c)
        assert F.encode(-mid) == (want | 0x80)
        # just off the tie goes to the nearer code
        assert F.encode(np.nextafter(mid, 0)) == c
        assert F.encode(np.nextafter(mid, 1e9)) == c + 1
    assert F.encode(460.0) == 0x7E  # would round to 480, which does not exist: saturate
    assert F.encode(1e30) == 0x7E and F.encode(-1e30) == 0xFE
    assert F.encode(np.inf) == 0x7E and F.encode(-np.inf) == 0xFE
    assert F.encode(np.nan) == 0x7F
    assert F.encode(2.0 ** -11) == 0x00  # below half the smallest subnormal
    assert F.encode(3 * 2.0 ** -11) == 0x01  # 0.75 quantum rounds up


def test_e4m3_encoder_agrees_with_torch_in_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.normal(0, 1, 20000),
        rng.normal(0, 100, 20000),
        rng.uniform(-448, 448, 20000),
        rng.normal(0, 2.0 ** -7, 20000),
    ]).astype(np.float32)
    x = x[np.abs(x) <= 448.0]  # torch's cast does not saturate; compare inside the finite range only
    t = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.encode(x.astype(np.float64)), t)


def test_quantize_rounds_the_product_in_float32():
    # the store multiplies by float32(1/scale) in float32 and encodes that product
    scale = 0.0123
    inv = np.float32(1.0) / np.float32(scale)
    x = np.linspace(-5, 5, 2001, dtype=np.float32)
    want = F.encode((x * inv).astype(np.float32).astype(np.float64))
    assert np.array_equal(F.quantize(x, scale), want)
    back = F.dequantize(F.quantize(x, scale), scale)
    # relative error of e4m3 is at most 2^-4 for normal values
    big = np.abs(x) > 2.0 ** -6 * scale * 2
    assert np.all(np.abs(back[big] - x[big]) <= np.abs(x[big]) * 2.0 ** -4 + 1e-12)
    # inputs whose float32 product lands exactly on the midpoint of two codes: there the rounding of
    # the product decides the code (ties to even), so a product taken in another precision shows
    d = F.decode_table()
    ties = []
    for c in range(0x08, 0x7E):  # consecutive normal codes c, c + 1
        t = np.float32((d[c] + d[c + 1]) / 2.0)
        x0 = np.float32(np.float64(t) / np.float64(inv))
        for k in range(-4, 5):
            xk = x0
            for _ in range(abs(k)):
                xk = np.nextafter(xk, np.float32(np.sign(k) * np.inf), dtype=np.float32)
            if np.float32(xk * inv) == t:
                ties.append((xk, c))
                break
    assert len(ties) > 60
    xt = np.array([v for v, _ in ties], dtype=np.float32)
    even = np.array([c if c % 2 == 0 else c + 1 for _, c in ties], dtype=np.uint8)
    assert np.array_equal(F.quantize(xt, scale), even)


def test_bf16_widening_is_exact():
    x = torch.randn(4096, dtype=torch.float32).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy()
    assert np.array_equal(A.bf16_bits_to_f64(bits), x.double().numpy())
    assert A.bf16_bits_to_f64(np.array([0x3F80], dtype=np.uint16))[0] == 1.0
    assert A.bf16_bits_to_f64(np.array([0xC000], dtype=np.uint16))[0] == -2.0


# ---------------------------------------------------------------------------------------------
# attention: independent restatements
# ---------------------------------------------------------------------------------------------
def _small_batch(seed, ps=4, Hq=4, Hkv=2, D=8, lens=((9, 1), (5, 5), (13, 4), (4, 2)), window=-1):
    """Random float64 pools and a CSR batch; every request owns random distinct pages."""
    rng = np.random.default_rng(seed)
    L = [a for a, _ in lens]
    n = [b for _, b in lens]
    counts = [(x + ps - 1) // ps for x in L]
    P = sum(counts) + 3
    perm = rng.permutation(P)
    rows, at = [], 0
    for c in counts:
        rows.append(perm[at:at + c])
        at += c
    kp = rng.normal(size=(P, ps, Hkv, D))
    vp = rng.normal(size=(P, ps, Hkv, D))
    q = rng.normal(size=(sum(n), Hq, D))
    qo = np.concatenate([[0], np.cumsum(n)])
    indptr = np.concatenate([[0], np.cumsum(counts)])
    indices = np.concatenate(rows)
    last = np.array([x - (c - 1) * ps for x, c in zip(L, counts)])
    return dict(q=q, k_pool=kp, v_pool=vp, qo_indptr=qo, kv_indptr=indptr, kv_indices=indices,
                last_page_len=last, page_size=ps, window_left=window), L, n


def _bruteforce(b, L, n, scale, causal=True):
    """Python loops only: walk each request's pages token by token, softmax with math.exp."""
    q, kp, vp, ps = b["q"], b["k_pool"], b["v_pool"], b["page_size"]
    Hq, D = q.shape[1], q.shape[2]
    Hkv = kp.shape[2]
    grp = Hq // Hkv
    w = b["window_left"]
    out = np.zeros_like(q)
    lse = np.zeros(q.shape[:2])
    for i in range(len(L)):
        pages = b["kv_indices"][b["kv_indptr"][i]:b["kv_indptr"][i + 1]]
        keys, vals = [], []
        for j in range(L[i]):
            keys.append(kp[pages[j // ps], j % ps])
            vals.append(vp[pages[j // ps], j % ps])
        for t in range(n[i]):
            row = b["qo_indptr"][i] + t
            pos = L[i] - n[i] + t
            for h in range(Hq):
                kh = h // grp
                js = [j for j in range(L[i]) if not causal or (j <= pos and (w < 0 or j >= pos - w))]
                s = [scale * sum(q[row, h, d] * keys[j][kh, d] for d in range(D)) for j in js]
                mx = max(s)
                e = [math.exp(x - mx) for x in s]
                den = math.fsum(e)
                for d in range(D):
                    out[row, h, d] = math.fsum(e[k] * vals[j][kh, d] for k, j in enumerate(js)) / den
                lse[row, h] = mx + math.log(den)
    return out, lse


def _oracle(b, scale, causal=True):
    return A.paged_attention(b["q"], b["k_pool"], b["v_pool"], b["qo_indptr"], b["kv_indptr"], b["kv_indices"],
                             b["last_page_len"], b["page_size"], sm_scale=scale, window_left=b["window_left"],
                             causal=causal)


def check_bruteforce(window=-1, seed=1, causal=True):
    lens = ((9, 1), (5, 5), (13, 4), (4, 2)) if causal else ((9, 1), (3, 5), (13, 4), (4, 2))  # non-causal: L < n allowed
    b, L, n = _small_batch(seed, window=window, lens=lens)
    scale = 0.37
    o, lse = _oracle(b, scale, causal=causal)
    bo, bl = _bruteforce(b, L, n, scale, causal=causal)
    return np.allclose(o, bo, rtol=0, atol=1e-12) and np.allclose(lse, bl, rtol=0, atol=1e-12)


def check_sdpa(window=-1, seed=2, causal=True):
    """The library routine the pages' CPU reference uses, in float64, with enable_gqa."""
    b, L, n = _small_batch(seed, ps=4, Hq=8, Hkv=2, D=16, window=window,
                           lens=((17, 3), (6, 6), (30, 1), (8, 0), (12, 7)))
    scale = 0.21
    o, _ = _oracle(b, scale, causal=causal)
    ps = b["page_size"]
    for i in range(len(L)):
        if n[i] == 0:
            continue
        pages = torch.from_numpy(b["kv_indices"][b["kv_indptr"][i]:b["kv_indptr"][i + 1]].astype(np.int64))
        k = torch.from_numpy(b["k_pool"])[pages].flatten(0, 1)[:L[i]].transpose(0, 1)
        v = torch.from_numpy(b["v_pool"])[pages].flatten(0, 1)[:L[i]].transpose(0, 1)
        q0, q1 = b["qo_indptr"][i], b["qo_indptr"][i + 1]
        qi = torch.from_numpy(b["q"][q0:q1]).transpose(0, 1)
        qpos = torch.arange(L[i] - n[i], L[i]).unsqueeze(1)
        kpos = torch.arange(L[i]).unsqueeze(0)
        mask = kpos <= qpos if causal else torch.ones((n[i], L[i]), dtype=torch.bool)
        if window >= 0:
            mask &= kpos >= qpos - window
        ref = torch.nn.functional.scaled_dot_product_attention(qi, k, v, attn_mask=mask, scale=scale, enable_gqa=True)
        if not np.allclose(o[q0:q1], ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12):
            return False
    return True


def check_page_size_one_view(seed=3):
    b, L, n = _small_batch(seed, ps=4)
    o, lse = _oracle(b, 0.5)
    ps = b["page_size"]
    p1, s1, l1 = M.to_page_size_one(b["kv_indptr"], b["kv_indices"], b["last_page_len"], ps)
    b1 = dict(b)
    P, _, H, D = b["k_pool"].shape
    b1.update(k_pool=b["k_pool"].reshape(P * ps, 1, H, D), v_pool=b["v_pool"].reshape(P * ps, 1, H, D),
              kv_indptr=p1, kv_indices=s1, last_page_len=l1, page_size=1)
    o1, lse1 = _oracle(b1, 0.5)
    return np.array_equal(o, o1) and np.array_equal(lse, lse1)


def check_page_permutation(seed=4):
    b, L, n = _small_batch(seed)
    o, _ = _oracle(b, 0.5)
    P = b["k_pool"].shape[0]
    perm = np.random.default_rng(seed).permutation(P)
    b2 = dict(b)
    kp2 = np.empty_like(b["k_pool"])
    vp2 = np.empty_like(b["v_pool"])
    kp2[perm] = b["k_pool"]
    vp2[perm] = b["v_pool"]
    b2.update(k_pool=kp2, v_pool=vp2, kv_indices=perm[b["kv_indices"]])
    o2, _ = _oracle(b2, 0.5)
    return np.array_equal(o, o2)


def check_single_key():
    rng = np.random.default_rng(5)
    ps, H, D = 4, 2, 8
    kp = rng.normal(size=(6, ps, H, D))
    vp = rng.normal(size=(6, ps, H, D))
    q = rng.normal(size=(3, H, D)) * 10
    # request 0: kv_len 1 decode; request 1: prefill with no prefix, first token sees only key 0
    o, _ = A.paged_attention(q, kp, vp, [0, 1, 3], [0, 1, 2], [4, 2], [1, 2], ps, sm_scale=1.0)
    ok = np.array_equal(o[0], vp[4, 0]) and np.array_equal(o[1], vp[2, 0])
    # window 0: only the query's own position is visible
    o2, _ = A.paged_attention(q[:1], kp, vp, [0, 1], [0, 3], [1, 3, 5], [2], ps, sm_scale=1.0, window_left=0)
    ok &= np.array_equal(o2[0], vp[5, 1])  # position 9 = page 2 (physical 5), offset 1
    return bool(ok)


def check_uniform_scores():
    b, L, n = _small_batch(6)
    b["q"] = np.zeros_like(b["q"])
    o, lse = _oracle(b, 0.9)
    ps = b["page_size"]
    grp = b["q"].shape[1] // b["k_pool"].shape[2]
    for i in range(len(L)):
        pages = b["kv_indices"][b["kv_indptr"][i]:b["kv_indptr"][i + 1]]
        for t in range(n[i]):
            pos = L[i] - n[i] + t
            vals = np.stack([b["v_pool"][pages[j // ps], j % ps] for j in range(pos + 1)])
            row = b["qo_indptr"][i] + t
            for h in range(b["q"].shape[1]):
                if not np.allclose(o[row, h], vals[:, h // grp].mean(axis=0), rtol=0, atol=1e-14):
                    return False
                if abs(lse[row, h] - math.log(pos + 1)) > 1e-12:
                    return False
    return True


def check_merge_closed_form(seed=7):
    rng = np.random.default_rng(seed)
    K = rng.normal(size=(50, 16))
    V = rng.normal(size=(50, 16))
    q = rng.normal(size=16) * 3
    o, s = A.attend(q, K, V, 0, 49, 0.4)
    for cut in (1, 17, 49):
        o1, s1 = A.attend(q, K, V, 0, cut - 1, 0.4)
        o2, s2 = A.attend(q, K, V, cut, 49, 0.4)
        om, sm = A.merge_states(o1, s1, o2, s2)
        if not (np.allclose(om, o, rtol=0, atol=1e-13) and abs(sm - s) < 1e-12):
            return False
    parts = [(0, 9), (10, 10), (11, 30), (31, 49)]
    res = [A.attend(q, K, V, a, b_, 0.4) for a, b_ in parts]
    om, sm = A.merge_many([r[0] for r in res], [r[1] for r in res])
    if not (np.allclose(om, o, rtol=0, atol=1e-13) and abs(sm - s) < 1e-12):
        return False
    # an empty state (lse = -inf) leaves the other unchanged
    oe, se = A.merge_states(np.zeros(16), -np.inf, o, s)
    return np.allclose(oe, o, rtol=0, atol=1e-15) and abs(se - s) < 1e-15


def check_prefix_suffix_merge(seed=8):
    """"SGLang 源码完全拆解(八)：Attention Backend", section «extend 的两种形态»: causal extend over a cached
    prefix of p keys plus n new keys = merge of (the n queries over the prefix, causal=False) and (the
    n queries over the n new keys alone, causal within the segment)."""
    rng = np.random.default_rng(seed)
    ps, Hq, Hkv, D = 4, 4, 2, 8
    for p_len, n in ((7, 3), (1, 6), (12, 1), (5, 5), (0, 4)):
        L = p_len + n
        P = (L + ps - 1) // ps + 2
        kp, vp = rng.normal(size=(P, ps, Hkv, D)), rng.normal(size=(P, ps, Hkv, D))
        q = rng.normal(size=(n, Hq, D)) * 2
        pages = rng.permutation(P)[: (L + ps - 1) // ps]
        full_o, full_s = A.paged_attention(q, kp, vp, [0, n], [0, len(pages)], pages,
                                           [L - (len(pages) - 1) * ps], ps, sm_scale=0.3)
        # prefix-only view: the first p keys (same pages, shorter length), every query sees all of them
        np_pre = (p_len + ps - 1) // ps  # 0 pages without a prefix: the empty state
        pre_o, pre_s = A.paged_attention(q, kp, vp, [0, n], [0, np_pre], pages[:np_pre],
                                         [p_len - (np_pre - 1) * ps if np_pre else 0], ps, sm_scale=0.3,
                                         causal=False)
        # suffix-only view: the n new keys as contiguous ("ragged") K/V, causal within the segment
        K = np.stack([kp[pages[j // ps], j % ps] for j in range(p_len, L)])
        V = np.stack([vp[pages[j // ps], j % ps] for j in range(p_len, L)])
        suf_o, suf_s = A.ragged_attention(q, K, V, [0, n], [0, n], sm_scale=0.3)
        mo, ms = A.merge_states(pre_o, pre_s, suf_o, suf_s)
        if not (np.allclose(mo, full_o, rtol=0, atol=1e-13) and np.allclose(ms, full_s, rtol=0, atol=1e-12)):
            return False
    return True


def _ragged_batch(seed, lens, Hq=4, Hkv=2, D=8):
    """Contiguous K/V rows per request (no page table): lens = ((kv_len, q_len), ...)."""
    rng = np.random.default_rng(seed)
    L = [a for a, _ in lens]
    n = [b_ for _, b_ in lens]
    k = rng.normal(size=(sum(L), Hkv, D))
    v = rng.normal(size=(sum(L), Hkv, D))
    q = rng.normal(size=(sum(n), Hq, D)) * 2
    return q, k, v, np.concatenate([[0], np.cumsum(n)]), np.concatenate([[0], np.cumsum(L)]), L, n


def check_ragged_bruteforce(seed=11, causal=True):
    """Python loops over each request's contiguous rows; a request with no keys must give (0, -inf)."""
    lens = ((6, 6), (9, 2), (3, 3), (5, 1)) if causal else ((6, 6), (2, 5), (0, 3), (5, 1))
    q, k, v, qo, kv, L, n = _ragged_batch(seed, lens)
    scale = 0.41
    o, lse = A.ragged_attention(q, k, v, qo, kv, sm_scale=scale, causal=causal)
    Hq, D = q.shape[1], q.shape[2]
    grp = Hq // k.shape[1]
    for i in range(len(L)):
        for t in range(n[i]):
            row = qo[i] + t
            pos = L[i] - n[i] + t
            js = [j for j in range(L[i]) if not causal or j <= pos]
            for h in range(Hq):
                if not js:
                    if not (np.all(o[row, h] == 0.0) and lse[row, h] == -math.inf):
                        return False
                    continue
                s = [scale * math.fsum(q[row, h, d] * k[kv[i] + j, h // grp, d] for d in range(D)) for j in js]
                mx = max(s)
                e = [math.exp(x - mx) for x in s]
                den = math.fsum(e)
                for d in range(D):
                    if abs(o[row, h, d] - math.fsum(e[a] * v[kv[i] + j, h // grp, d] for a, j in enumerate(js)) / den) > 1e-12:
                        return False
                if abs(lse[row, h] - (mx + math.log(den))) > 1e-12:
                    return False
    return True


def check_ragged_sdpa(seed=12):
    """Causal self-attention over a fresh segment (n == kv_len) is SDPA's is_causal form."""
    q, k, v, qo, kv, L, n = _ragged_batch(seed, ((7, 7), (1, 1), (12, 12)), Hq=8, Hkv=2, D=16)
    o, _ = A.ragged_attention(q, k, v, qo, kv, sm_scale=0.23)
    for i in range(len(L)):
        qi = torch.from_numpy(q[qo[i]:qo[i + 1]]).transpose(0, 1)
        ki = torch.from_numpy(k[kv[i]:kv[i + 1]]).transpose(0, 1)
        vi = torch.from_numpy(v[kv[i]:kv[i + 1]]).transpose(0, 1)
        ref = torch.nn.functional.scaled_dot_product_attention(qi, ki, vi, is_causal=True, scale=0.23, enable_gqa=True)
        if not np.allclose(o[qo[i]:qo[i + 1]], ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12):
            return False
    return True


def test_ragged_bruteforce_causal():
    assert check_ragged_bruteforce()


def test_ragged_bruteforce_noncausal_and_empty_segment():
    assert check_ragged_bruteforce(causal=False)


def test_ragged_matches_library_sdpa_is_causal():
    assert check_ragged_sdpa()


def test_noncausal_paged_segment_without_keys_is_the_empty_state():
    b, L, n = _small_batch(13, lens=((5, 2), (0, 3), (4, 4)))
    o, lse = _oracle(b, 0.5, causal=False)
    r = slice(b["qo_indptr"][1], b["qo_indptr"][2])
    assert np.all(o[r] == 0.0) and np.all(lse[r] == -np.inf)
    assert np.all(np.isfinite(lse[: b["qo_indptr"][1]]))


def check_cascade_shared_prefix(seed=14):
    """"vLLM 源码完全拆解（六）：Attention Backend", section «Cascade Attention 把共享前缀只算一次»: when the
    requests of a batch share a prefix, each query's attention splits into the shared prefix (computed
    once for all queries: one "request" holding every query row, all prefix keys visible) and its own
    suffix (causal), merged by their LSE weights -- equal to each request's flat causal pass."""
    rng = np.random.default_rng(seed)
    ps, Hq, Hkv, D = 4, 4, 2, 8
    shared_pages = 3
    suffix = [5, 1, 9, 4]
    n = [1, 1, 3, 4]
    Lp = shared_pages * ps
    own = [(x + ps - 1) // ps for x in suffix]
    P = shared_pages + sum(own) + 2
    kp, vp = rng.normal(size=(P, ps, Hkv, D)), rng.normal(size=(P, ps, Hkv, D))
    perm = rng.permutation(P)
    shared = perm[:shared_pages]
    rows, at = [], shared_pages
    for c in own:
        rows.append(perm[at:at + c])
        at += c
    q = rng.normal(size=(sum(n), Hq, D)) * 2
    qo = np.concatenate([[0], np.cumsum(n)])
    last = [x - (c - 1) * ps for x, c in zip(suffix, own)]
    # flat: every request's page list = shared pages + its own pages
    flat_ptr = np.concatenate([[0], np.cumsum([shared_pages + c for c in own])])
    flat_idx = np.concatenate([np.concatenate([shared, r]) for r in rows])
    fo, fs = A.paged_attention(q, kp, vp, qo, flat_ptr, flat_idx, last, ps, sm_scale=0.35)
    # level 0: all query rows as one request over the shared pages, non-causal
    so, ss = A.paged_attention(q, kp, vp, [0, qo[-1]], [0, shared_pages], shared, [ps], ps, sm_scale=0.35,
                               causal=False)
    # level 1: each request over its own suffix pages, causal
    uo, us = A.paged_attention(q, kp, vp, qo, np.concatenate([[0], np.cumsum(own)]), np.concatenate(rows), last, ps,
                               sm_scale=0.35)
    mo, ms = A.merge_states(so, ss, uo, us)
    assert Lp == 12
    return bool(np.allclose(mo, fo, rtol=0, atol=1e-13) and np.allclose(ms, fs, rtol=0, atol=1e-12))


def test_cascade_shared_prefix_merge_equals_flat_causal():
    assert check_cascade_shared_prefix()


def test_bruteforce_tiny():
    assert check_bruteforce()


def test_bruteforce_tiny_noncausal():
    assert check_bruteforce(causal=False)


def test_matches_library_sdpa_noncausal():
    assert check_sdpa(causal=False)


def test_prefix_noncausal_merged_with_causal_suffix_equals_causal_extend():
    assert check_prefix_suffix_merge()


def test_noncausal_rejects_a_window():
    b, L, n = _small_batch(1, window=2)
    with pytest.raises(ValueError):
        _oracle(b, 0.5, causal=False)


def test_bruteforce_tiny_window():
    assert check_bruteforce(window=3)


def test_matches_library_sdpa_with_gqa():
    assert check_sdpa()


def test_matches_library_sdpa_with_window():
    assert check_sdpa(window=5)


def test_page_size_one_view_is_identical():
    assert check_page_size_one_view()


def test_physical_page_permutation_is_invisible():
    assert check_page_permutation()


def test_single_visible_key_returns_v():
    assert check_single_key()


def test_uniform_scores_return_mean_v():
    assert check_uniform_scores()


def test_split_and_merge_equals_unsplit():
    assert check_merge_closed_form()


def test_kv_store_scatter_and_padding():
    g = _golden("vllm_worked_example.json")
    ps = 16
    sm = M.slot_mapping(g["block_table"], g["query_start_loc"], g["seq_lens"], ps)
    sm = np.concatenate([sm, [-1]])  # a padding token
    kp = np.zeros((13, ps, 2, 4))
    vp = np.zeros((13, ps, 2, 4))
    k = np.arange(9 * 8, dtype=np.float64).reshape(9, 2, 4) + 1
    v = -k
    A.kv_store(kp, vp, k, v, sm, ps)
    assert np.array_equal(kp[10, 15], k[0])  # slot 175
    assert np.array_equal(kp[5, 0:4], k[1:5])  # slots 80..83
    assert np.array_equal(vp[12, 0:3], v[5:8])  # slots 192..194
    assert np.count_nonzero(kp) == 8 * 8  # the padding row wrote nothing


def test_write_before_read_decode_sees_its_own_token():
    b, L, n = _small_batch(8, lens=((9, 1), (4, 1)))
    # make the query point strongly along the new key so the new token dominates
    ps = b["page_size"]
    knew = np.random.default_rng(9).normal(size=(2, 2, 8))
    vnew = np.random.default_rng(10).normal(size=(2, 2, 8))
    slots = []
    for i in range(2):
        pages = b["kv_indices"][b["kv_indptr"][i]:b["kv_indptr"][i + 1]]
        pos = L[i] - 1
        slots.append(pages[pos // ps] * ps + pos % ps)
    A.kv_store(b["k_pool"], b["v_pool"], knew, vnew, slots, ps)
    grp = b["q"].shape[1] // 2
    for i in range(2):
        for h in range(b["q"].shape[1]):
            b["q"][i, h] = 60.0 * knew[i, h // grp]
    o, _ = _oracle(b, 1.0)
    for i in range(2):
        for h in range(b["q"].shape[1]):
            assert np.allclose(o[i, h], vnew[i, h // grp], atol=1e-6)


def test_rejects_kv_shorter_than_queries():
    b, L, n = _small_batch(11)
    b["qo_indptr"] = np.array([0, 1, 20, 24, 26])  # request 1 claims 19 queries but has 5 keys
    b["q"] = np.zeros((26, 4, 8))
    with pytest.raises(ValueError):
        _oracle(b, 1.0)
