"""Paged-KV metadata, restated from the pages (oracle; test infrastructure only).

Sources:

* "vLLM 源码完全拆解（六）：Attention Backend", sections «Runner 先构造公共事实»
  (the worked slot_mapping example), «从二维 Block Table 到 CSR 页表» (page
  count, indptr and last-page-length; a remainder of 0 means a full page, not
  an empty one) and «FlashInfer Builder 的结果» (the worked CSR example and the
  decode-first split of qo_indptr).
* "SGLang 源码完全拆解(八)：Attention Backend", section «统一元数据的编译»: the
  three CSR arrays and what each one means.
* "手写 mini-sglang 阶段四 · GPU 注意力后端", sections «FlashAttention：页号表»
  (page ids are the token table sampled every page_size entries, divided by
  page_size), «把 KV 池当成 page size = 1» and the exercise answer (page count
  ``ceil(len / ps)``, ``last_page_len = len - (pages - 1) * ps``).

All functions take and return plain numpy integer arrays.
"""

from __future__ import annotations

import numpy as np


def num_pages_for(seq_len: int, page_size: int) -> int:
    """Pages a request of ``seq_len`` tokens occupies: ceil(seq_len / page_size)."""
    if seq_len < 0 or page_size < 1:
        raise ValueError("seq_len must be >= 0 and page_size >= 1")
    return (seq_len + page_size - 1) // page_size


def last_page_len_for(seq_len: int, page_size: int) -> int:
    """Valid tokens on the last page: seq_len - (pages - 1) * page_size, in [1, page_size].

    A remainder of zero is a FULL last page (page_size), never 0.
    """
    n = num_pages_for(seq_len, page_size)
    if n == 0:
        raise ValueError("a request with no tokens has no last page")
    return seq_len - (n - 1) * page_size


def slot_of(block_row, position: int, page_size: int) -> int:
    """KV write address of one token: physical_page * page_size + offset_in_page.

    ``block_row`` is the request's row of the 2-D block table (physical page id
    of each logical page); ``position`` is the token's absolute position in the
    request.
    """
    logical_page = position // page_size
    offset = position % page_size
    return int(block_row[logical_page]) * page_size + offset


def slot_mapping(block_table, query_start_loc, seq_lens, page_size: int) -> np.ndarray:
    """Per-token write slots for a flat batch of new tokens.

    Request i contributes ``query_start_loc[i+1] - query_start_loc[i]`` new
    tokens; they are its LAST positions, ``seq_lens[i] - n_i ... seq_lens[i] - 1``.
    """
    out = []
    for i in range(len(seq_lens)):
        n = int(query_start_loc[i + 1] - query_start_loc[i])
        L = int(seq_lens[i])
        for pos in range(L - n, L):
            out.append(slot_of(block_table[i], pos, page_size))
    return np.asarray(out, dtype=np.int64)


def csr_from_block_table(block_table, seq_lens, page_size: int):
    """2-D block table -> CSR page table (kv_indptr, kv_indices, last_page_len).

    kv_indptr is the prefix sum of per-request page counts; kv_indices
    concatenates the first ``pages_i`` valid physical ids of every row;
    last_page_len is the fill of each request's final page.
    """
    counts = [num_pages_for(int(L), page_size) for L in seq_lens]
    kv_indptr = np.zeros(len(seq_lens) + 1, dtype=np.int64)
    kv_indptr[1:] = np.cumsum(counts)
    kv_indices = []
    for i, c in enumerate(counts):
        kv_indices.extend(int(p) for p in block_table[i][:c])
    last = [last_page_len_for(int(L), page_size) for L in seq_lens]
    return kv_indptr, np.asarray(kv_indices, dtype=np.int64), np.asarray(last, dtype=np.int64)


def kv_lens_from_csr(kv_indptr, last_page_len, page_size: int) -> np.ndarray:
    """Inverse of the CSR encoding: L_i = (pages_i - 1) * page_size + last_page_len_i (0 if no pages)."""
    out = []
    for i in range(len(kv_indptr) - 1):
        n = int(kv_indptr[i + 1] - kv_indptr[i])
        out.append(0 if n == 0 else (n - 1) * page_size + int(last_page_len[i]))
    return np.asarray(out, dtype=np.int64)


def page_table_from_token_table(token_table, seq_lens, page_size: int) -> np.ndarray:
    """Token-granular table -> page ids: row[:max_len:page_size] // page_size.

    Every row is sampled up to the longest sequence of the batch (rows are
    padded the same way the page's FlashAttention path pads them).
    """
    max_len = int(max(seq_lens))
    rows = [np.asarray(token_table[i][:max_len:page_size]) // page_size for i in range(len(seq_lens))]
    return np.stack(rows).astype(np.int64)


def token_csr_from_token_table(token_table, seq_lens):
    """The page-size-1 view: kv_indices are token slots, last_page_len is all ones."""
    kv_indptr = np.zeros(len(seq_lens) + 1, dtype=np.int64)
    kv_indptr[1:] = np.cumsum([int(L) for L in seq_lens])
    kv_indices = np.concatenate([np.asarray(token_table[i][: int(L)]) for i, L in enumerate(seq_lens)])
    return kv_indptr, kv_indices.astype(np.int64), np.ones(len(seq_lens), dtype=np.int64)


def to_page_size_one(kv_indptr, kv_indices, last_page_len, page_size: int):
    """Re-express a page-granular CSR batch as the equivalent page-size-1 (token slot) batch.

    A pool of shape [P, ps, H, D] viewed as [P * ps, 1, H, D] holds logical
    token j of request i at slot kv_indices[kv_indptr[i] + j // ps] * ps + j % ps.
    """
    lens = kv_lens_from_csr(kv_indptr, last_page_len, page_size)
    slots = []
    indptr = np.zeros(len(lens) + 1, dtype=np.int64)
    for i, L in enumerate(lens):
        pages = kv_indices[kv_indptr[i] : kv_indptr[i + 1]]
        for j in range(int(L)):
            slots.append(int(pages[j // page_size]) * page_size + j % page_size)
        indptr[i + 1] = indptr[i] + int(L)
    return indptr, np.asarray(slots, dtype=np.int64), np.ones(len(lens), dtype=np.int64)


def decode_first_split(query_start_loc, threshold: int = 1):
    """Split a batch that is already ordered decode-first into its two slices.

    Requests whose query length is <= threshold form the decode slice; the rest
    form the prefill slice, whose qo_indptr is re-based to start at 0.
    Returns (num_decodes, num_decode_tokens, num_prefills, num_prefill_tokens,
    prefill_qo_indptr).
    """
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    qlen = np.diff(qsl)
    nd = 0
    while nd < len(qlen) and qlen[nd] <= threshold:
        nd += 1
    if np.any(qlen[nd:] <= threshold):
        raise ValueError("batch is not ordered decode-first")
    prefill = qsl[nd:] - qsl[nd]
    return nd, int(qsl[nd]), len(qlen) - nd, int(qsl[-1] - qsl[nd]), prefill
