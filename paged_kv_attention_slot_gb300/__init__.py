"""Batched attention over a paged KV cache on GB300 (sm_103a): Python binding of libpkv_attn.so.

The binding only marshals arguments; every step of the path (the KV write, the plan's device
copy, decode, split-KV merge, prefill) runs in the library's CUDA kernels.  PyTorch supplies
device memory and the current stream.

Typical use (plan once per batch, run once per layer):

    cache = KVCache(k_pool, v_pool)                     # [pages, page_size, kv_heads, head_dim]
    kv_store(k_new, v_new, slot_mapping, cache)         # write this step's tokens first
    plan = Plan()
    plan.plan(qo_indptr, kv_indptr, kv_indices, last_page_len,
              num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16, mode="decode")
    out, lse = plan.run(q, cache, return_lse=True)

Prefix-cached extend in the paged + merge form (new tokens' K/V read directly, the cached prefix
through the page table with every prefix key visible, the two states merged by their LSE):

    rag = Plan().plan(qo_indptr, qo_indptr, None, None, ..., mode="ragged")       # causal
    pre = Plan().plan(qo_indptr, pre_indptr, pre_indices, pre_last, ..., mode="prefill", causal=False)
    o1, s1 = rag.run_ragged(q, k_new, v_new, return_lse=True)
    o2, s2 = pre.run(q, cache, return_lse=True)
    out, lse = merge_state(o1, s1, o2, s2)
"""

from __future__ import annotations

import ctypes as C

import numpy as np
import torch

from . import _lib
from ._lib import PkvError, check, lib

__all__ = [
    "KVCache", "Plan", "CascadePlan", "PkvError", "kv_store", "merge_state", "device_error", "block_table_to_csr",
    "token_table_to_page_table", "library_path",
]


def library_path() -> str:
    return _lib.LIB_PATH


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_ptr(stream) -> int:
    """cudaStream_t of `stream`, or of the current stream on the current device."""
    if stream is not None:
        return int(stream.cuda_stream)
    if _raw_stream is not None:  # the current stream's handle without building a Stream object
        return int(_raw_stream(torch.cuda.current_device()))
    return int(torch.cuda.current_stream().cuda_stream)


def _i32(a) -> np.ndarray:
    if isinstance(a, np.ndarray) and a.dtype == np.int32 and a.flags.c_contiguous:
        return a  # already what the C ABI reads: no copy
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


_EMPTY_I32 = np.zeros(1, dtype=np.int32)  # a valid address for optional arrays that are absent


def _addr(a: np.ndarray) -> int:
    """Address of a C-contiguous array's data (the buffer route is ~4x cheaper than .ctypes.data)."""
    try:
        return C.addressof(C.c_int32.from_buffer(a))
    except (TypeError, ValueError):  # read-only or empty arrays
        return a.ctypes.data


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(C.POINTER(C.c_int32))


class KVCache:
    """One layer's K and V pools, [num_pages, page_size, num_kv_heads, head_dim].

    bf16 pools are torch.bfloat16 tensors; FP8 pools are torch.uint8 (or float8_e4m3fn) tensors of
    E4M3 codes with k_scale / v_scale (real value = code * scale).  The last dimension must be
    contiguous; other strides are passed through as they are.
    """

    def __init__(self, k: torch.Tensor, v: torch.Tensor, k_scale: float = 1.0, v_scale: float = 1.0):
        if k.shape != v.shape or k.dim() != 4:
            raise ValueError("k and v pools must both be [num_pages, page_size, num_kv_heads, head_dim]")
        if k.stride() != v.stride():
            raise ValueError("k and v pools must share strides")
        if k.stride(3) != 1:
            raise ValueError("head_dim must be the contiguous dimension")
        if k.dtype == torch.bfloat16:
            dtype = _lib.PKV_BF16
        elif k.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", None)):
            dtype = _lib.PKV_FP8_E4M3
        else:
            raise ValueError(f"unsupported pool dtype {k.dtype}")
        if v.dtype != k.dtype:
            raise ValueError("k and v pools must have the same dtype")
        self.k, self.v = k, v
        self.k_scale, self.v_scale = float(k_scale), float(v_scale)
        self.dtype = dtype
        self.struct = _lib.pkv_cache(
            k.data_ptr(), v.data_ptr(), k.shape[0], k.shape[1], k.shape[2], k.shape[3], dtype,
            k.stride(0), k.stride(1), k.stride(2), self.k_scale, self.v_scale)

    @property
    def num_pages(self):
        return self.k.shape[0]

    @property
    def page_size(self):
        return self.k.shape[1]

    @property
    def num_kv_heads(self):
        return self.k.shape[2]

    @property
    def head_dim(self):
        return self.k.shape[3]


def kv_store(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, cache: KVCache, stream=None) -> None:
    """Write k, v ([T, num_kv_heads, head_dim] bf16, contiguous) at slot_mapping ([T] int64, device)."""
    if k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise ValueError("k and v must be bf16")
    if not (k.is_contiguous() and v.is_contiguous() and slot_mapping.is_contiguous()):
        raise ValueError("k, v and slot_mapping must be contiguous")
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    T = k.shape[0]
    if v.shape != k.shape or slot_mapping.shape[0] != T or tuple(k.shape[1:]) != (cache.num_kv_heads, cache.head_dim):
        raise ValueError("shape mismatch between k, v, slot_mapping and the cache")
    check(lib().pkv_kv_store(k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), T, C.byref(cache.struct),
                             _stream_ptr(stream)))


def device_error(reset: bool = True, stream=None) -> int:
    """Synchronise and read (and by default clear) the device error word; 0 means no error."""
    code = C.c_int32(0)
    st = lib().pkv_device_error(C.byref(code), 1 if reset else 0, _stream_ptr(stream))
    if st not in (_lib.PKV_OK, _lib.PKV_EDEVICE):
        check(st)
    return int(code.value)


def set_wait_limit(clock_cycles: int = 0) -> None:
    """Bound, in SM clock cycles, on each wait inside the prefill kernel for runs launched from now
    on (0 restores the default, about 2 s).  A wait that runs out records PKV_DEVERR_TIMEOUT (read by
    device_error()) and its CTA exits without writing its rows."""
    check(lib().pkv_set_wait_limit(int(clock_cycles)))


_MODES = {"decode": _lib.PKV_MODE_DECODE, "prefill": _lib.PKV_MODE_PREFILL, "extend": _lib.PKV_MODE_PREFILL,
          "mixed": _lib.PKV_MODE_MIXED, "ragged": _lib.PKV_MODE_RAGGED, "paged_ragged": _lib.PKV_MODE_PAGED_RAGGED}
_KV_DTYPES = {"bf16": _lib.PKV_BF16, "e4m3": _lib.PKV_FP8_E4M3, "fp8": _lib.PKV_FP8_E4M3}


class Plan:
    """A reusable plan object: plan() once per batch, run() once per layer."""

    def __init__(self):
        h = C.c_void_p()
        check(lib().pkv_plan_create(C.byref(h)))
        self._h = h
        self.workspace = None
        self.mode = None
        self._keep = None

    def __del__(self):
        try:
            if getattr(self, "_h", None) is not None and self._h.value:
                lib().pkv_plan_destroy(self._h)
                self._h = None
        except Exception:
            pass

    @staticmethod
    def _args(qo_indptr, kv_indptr, kv_indices, last_page_len, num_qo_heads, num_kv_heads, head_dim, page_size,
              mode, window_left, sm_scale, kv_dtype, max_splits, num_sms, causal=True):
        # ragged plans have no page table: kv_indices / last_page_len may be None
        arrs = [_i32(qo_indptr), _i32(kv_indptr), _EMPTY_I32 if kv_indices is None else _i32(kv_indices),
                _EMPTY_I32 if last_page_len is None else _i32(last_page_len)]
        B = len(arrs[0]) - 1
        a = _lib.pkv_plan_args(B, _addr(arrs[0]), _addr(arrs[1]), _addr(arrs[2]), _addr(arrs[3]), num_qo_heads,
                               num_kv_heads, head_dim, page_size, _MODES[mode], 1 if causal else 0, window_left,
                               float(sm_scale), _lib.PKV_BF16, _KV_DTYPES[kv_dtype], max_splits, num_sms)
        return a, arrs

    @staticmethod
    def workspace_size(qo_indptr, kv_indptr, kv_indices, last_page_len, *, num_qo_heads, num_kv_heads, head_dim,
                       page_size=1, mode="decode", window_left=-1, sm_scale=0.0, kv_dtype="bf16", max_splits=0,
                       num_sms=0, causal=True) -> int:
        a, keep = Plan._args(qo_indptr, kv_indptr, kv_indices, last_page_len, num_qo_heads, num_kv_heads,
                             head_dim, page_size, mode, window_left, sm_scale, kv_dtype, max_splits, num_sms, causal)
        n = C.c_size_t(0)
        check(lib().pkv_plan_workspace_size(C.byref(a), C.byref(n)))
        return int(n.value)

    def plan(self, qo_indptr, kv_indptr, kv_indices, last_page_len, *, num_qo_heads, num_kv_heads, head_dim,
             page_size=1, mode="decode", window_left=-1, sm_scale=0.0, kv_dtype="bf16", max_splits=0, num_sms=0,
             causal=True, workspace: torch.Tensor | None = None, host_only: bool = False, stream=None) -> "Plan":
        """Plan a batch.  Host int arrays in; the binding keeps a device workspace (grown on demand).

        mode "ragged": kv_indptr holds row offsets into contiguous k / v tensors (run with
        run_ragged); kv_indices, last_page_len and page_size are ignored.  causal=False: every query
        sees all keys of its request (prefill / ragged plans)."""
        a, keep = self._args(qo_indptr, kv_indptr, kv_indices, last_page_len, num_qo_heads, num_kv_heads, head_dim,
                             page_size, mode, window_left, sm_scale, kv_dtype, max_splits, num_sms, causal)
        if host_only:
            check(lib().pkv_attn_plan(self._h, C.byref(a), None, 0, None))
        else:
            if workspace is not None:
                self.workspace = workspace
            if self.workspace is None:
                self.workspace = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
            st = lib().pkv_attn_plan(self._h, C.byref(a), self.workspace.data_ptr(), self.workspace.numel(),
                                     _stream_ptr(stream))
            if st == _lib.PKV_EWORKSPACE and workspace is None:
                # grow the binding-owned workspace and plan again
                n = C.c_size_t(0)
                check(lib().pkv_plan_workspace_size(C.byref(a), C.byref(n)))
                self.workspace = torch.empty(int(n.value) + (int(n.value) >> 2), dtype=torch.uint8, device="cuda")
                st = lib().pkv_attn_plan(self._h, C.byref(a), self.workspace.data_ptr(), self.workspace.numel(),
                                         _stream_ptr(stream))
            check(st)
        self.mode = mode
        self.num_qo_heads = num_qo_heads
        self.head_dim = head_dim
        self.total_tokens = int(keep[0][-1]) if len(keep[0]) else 0
        self.kv_rows = int(keep[1][-1]) if (mode == "ragged" and len(keep[1])) else 0
        self.num_kv_heads = num_kv_heads
        self._keep = keep
        return self

    def info(self) -> dict:
        i = _lib.pkv_plan_info()
        check(lib().pkv_plan_info_get(self._h, C.byref(i)))
        return {f: getattr(i, f) for f, _ in i._fields_}

    def work_items(self) -> np.ndarray:
        n = self.info()["num_work"]
        out = np.zeros(max(n, 1) * 8, dtype=np.int32)
        check(lib().pkv_plan_work_items(self._h, _ptr(out), out.size))
        return out[: n * 8].reshape(n, 8)

    def _outputs(self, q, out, lse, return_lse):
        if q.dtype != torch.bfloat16 or not q.is_contiguous():
            raise ValueError("q must be a contiguous bf16 tensor")
        if tuple(q.shape) != (self.total_tokens, self.num_qo_heads, self.head_dim):
            raise ValueError(f"q must be [{self.total_tokens}, {self.num_qo_heads}, {self.head_dim}]")
        if out is None:
            out = torch.empty_like(q)
        if (return_lse or lse is not None) and lse is None:
            lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
        return out, lse

    def run_ragged(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor | None = None,
                   lse: torch.Tensor | None = None, return_lse: bool = False, stream=None):
        """Attention of a "ragged" plan: k, v are contiguous bf16 [kv_indptr[-1], num_kv_heads, head_dim]."""
        if self.mode != "ragged":
            raise ValueError("run_ragged needs a plan made with mode='ragged'")
        for name, t in (("k", k), ("v", v)):
            if t.dtype != torch.bfloat16 or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous bf16 tensor")
            if tuple(t.shape) != (self.kv_rows, self.num_kv_heads, self.head_dim):
                raise ValueError(f"{name} must be [{self.kv_rows}, {self.num_kv_heads}, {self.head_dim}]")
        out, lse = self._outputs(q, out, lse, return_lse)
        check(lib().pkv_attn_ragged_run(self._h, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                        lse.data_ptr() if lse is not None else None, _stream_ptr(stream)))
        return (out, lse) if (return_lse or lse is not None) else out

    def run_paged_ragged(self, q: torch.Tensor, cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor,
                         out: torch.Tensor | None = None, lse: torch.Tensor | None = None, return_lse: bool = False,
                         stream=None):
        """Attention of a "paged_ragged" plan in one pass: the page table holds each request's cached
        prefix in `cache`; k_new, v_new are contiguous bf16 [total_tokens, num_kv_heads, head_dim] holding
        the new tokens' K / V (row r = token r of q)."""
        if self.mode != "paged_ragged":
            raise ValueError("run_paged_ragged needs a plan made with mode='paged_ragged'")
        for name, t in (("k_new", k_new), ("v_new", v_new)):
            if t.dtype != torch.bfloat16 or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous bf16 tensor")
            if tuple(t.shape) != (self.total_tokens, self.num_kv_heads, self.head_dim):
                raise ValueError(f"{name} must be [{self.total_tokens}, {self.num_kv_heads}, {self.head_dim}]")
        out, lse = self._outputs(q, out, lse, return_lse)
        check(lib().pkv_attn_paged_ragged_run(self._h, q.data_ptr(), C.byref(cache.struct), k_new.data_ptr(),
                                              v_new.data_ptr(), out.data_ptr(),
                                              lse.data_ptr() if lse is not None else None, _stream_ptr(stream)))
        return (out, lse) if (return_lse or lse is not None) else out

    def run(self, q: torch.Tensor, cache: KVCache, out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
            return_lse: bool = False, merge_into: bool = False, stream=None):
        """Attention for every planned token row; q is [total_tokens, num_qo_heads, head_dim] bf16.

        merge_into=True (prefill plans): out / lse hold a state on entry (e.g. from run_ragged over the
        new tokens) and receive the merge of that state with this pass's (pkv_attn_prefill_run_merge)."""
        if self.mode == "ragged":
            raise ValueError("a ragged plan runs with run_ragged(q, k, v)")
        if self.mode == "paged_ragged":
            raise ValueError("a paged_ragged plan runs with run_paged_ragged(q, cache, k_new, v_new)")
        if merge_into:
            if self.mode not in ("prefill", "extend") or out is None or lse is None:
                raise ValueError("merge_into needs a prefill plan and the held state in out and lse")
            self._outputs(q, out, lse, True)
            check(lib().pkv_attn_prefill_run_merge(self._h, q.data_ptr(), C.byref(cache.struct), out.data_ptr(),
                                                   lse.data_ptr(), _stream_ptr(stream)))
            return out, lse
        out, lse = self._outputs(q, out, lse, return_lse)
        if self.mode == "decode":
            fns = [lib().pkv_attn_decode_run]
        elif self.mode == "mixed":  # one-token rows on the decode kernel, the rest on the prefill kernel
            fns = [lib().pkv_attn_decode_run, lib().pkv_attn_prefill_run]
        else:
            fns = [lib().pkv_attn_prefill_run]
        for fn in fns:
            check(fn(self._h, q.data_ptr(), C.byref(cache.struct), out.data_ptr(),
                     lse.data_ptr() if lse is not None else None, _stream_ptr(stream)))
        return (out, lse) if (return_lse or lse is not None) else out


class CascadePlan:
    """Attention for a batch whose requests share a prefix, with the shared part computed once.

    "vLLM 源码完全拆解（六）：Attention Backend", section «Cascade Attention 把共享前缀只算一次»: each
    query's attention is split into the shared prefix and its request's own suffix, and the two
    outputs are combined by their log-sum-exp weights.  Level 0 is one non-causal prefill plan in
    which a single "request" holds every query row of the batch and the shared pages (so each
    shared K/V tile is read once per query tile instead of once per request); level 1 is an ordinary
    causal plan over each request's own suffix pages (decode when every request has one new token).
    The run is one library call, pkv_cascade_run: level 1 into ``out``/``lse``, then level 0 with
    its state merged into them in its epilogue.
    """

    def __init__(self):
        self.shared = Plan()
        self.suffix = Plan()

    def plan(self, qo_indptr, shared_kv_indices, shared_last_page_len: int, kv_indptr, kv_indices, last_page_len, *,
             num_qo_heads, num_kv_heads, head_dim, page_size, sm_scale=0.0, num_sms=0, max_splits=0,
             stream=None) -> "CascadePlan":
        """shared_kv_indices: the shared prefix's pages in order (its last page holds
        shared_last_page_len tokens); kv_indptr / kv_indices / last_page_len: each request's own
        suffix pages (the suffix holds the new tokens, so every request with a new token has one)."""
        qo = _i32(qo_indptr)
        shared = _i32(shared_kv_indices)
        kw = dict(num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads, head_dim=head_dim, page_size=page_size,
                  sm_scale=sm_scale, num_sms=num_sms, max_splits=max_splits, stream=stream)
        T = int(qo[-1]) if len(qo) else 0
        self.shared.plan([0, T], [0, len(shared)], shared, [shared_last_page_len if len(shared) else 0],
                         mode="prefill", causal=False, **kw)
        n = np.diff(qo)
        mode = "decode" if np.all(n <= 1) else ("mixed" if np.any(n == 1) else "prefill")
        self.suffix.plan(qo, kv_indptr, kv_indices, last_page_len, mode=mode, **kw)
        self.total_tokens = T
        return self

    def run(self, q: torch.Tensor, cache: KVCache, out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
            return_lse: bool = False, stream=None):
        """pkv_cascade_run: the suffix plan into (out, lse), then the shared pass merged into them."""
        if lse is None:
            lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
        out, lse = self.suffix._outputs(q, out, lse, True)
        check(lib().pkv_cascade_run(self.shared._h, self.suffix._h, q.data_ptr(), C.byref(cache.struct),
                                    out.data_ptr(), lse.data_ptr(), _stream_ptr(stream)))
        return (out, lse) if return_lse else out


def merge_state(o_a: torch.Tensor, lse_a: torch.Tensor, o_b: torch.Tensor, lse_b: torch.Tensor,
                out: torch.Tensor | None = None, lse_out: torch.Tensor | None = None, stream=None):
    """Merge two attention states of the same rows by their log-sum-exp (natural log).

    o_*: bf16 [..., head_dim] contiguous; lse_*: float32 with o's shape minus the last dimension.
    out / lse_out may be o_a / lse_a (in place).  Returns (out, lse_out)."""
    if o_a.shape != o_b.shape or lse_a.shape != lse_b.shape or tuple(lse_a.shape) != tuple(o_a.shape[:-1]):
        raise ValueError("o_a, o_b must share a shape and lse_a, lse_b must be that shape without head_dim")
    for t in (o_a, o_b):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("o_a and o_b must be contiguous bf16 tensors")
    for t in (lse_a, lse_b):
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError("lse_a and lse_b must be contiguous float32 tensors")
    if out is None:
        out = torch.empty_like(o_a)
    if lse_out is None:
        lse_out = torch.empty_like(lse_a)
    check(lib().pkv_merge_state(o_a.data_ptr(), lse_a.data_ptr(), o_b.data_ptr(), lse_b.data_ptr(), out.data_ptr(),
                                lse_out.data_ptr(), lse_a.numel(), o_a.shape[-1], _stream_ptr(stream)))
    return out, lse_out


def block_table_to_csr(block_table, seq_lens, page_size: int):
    """Host helper: 2-D block table -> (kv_indptr, kv_indices, last_page_len) int32 numpy arrays."""
    bt = _i32(block_table)
    sl = _i32(seq_lens)
    B, W = bt.shape
    indptr = np.zeros(B + 1, dtype=np.int32)
    cap = max(1, B * W)
    indices = np.zeros(cap, dtype=np.int32)
    last = np.zeros(B, dtype=np.int32)
    check(lib().pkv_block_table_to_csr(_ptr(bt), B, W, _ptr(sl), page_size, _ptr(indptr), _ptr(indices), cap,
                                       _ptr(last)))
    return indptr, indices[: indptr[-1]].copy(), last


def token_table_to_page_table(token_table, seq_lens, page_size: int):
    """Host helper: token-granular table -> page table (row[:max_len:page_size] // page_size)."""
    tt = _i32(token_table)
    sl = _i32(seq_lens)
    B, W = tt.shape
    cols = (int(sl.max()) + page_size - 1) // page_size if B else 0
    out = np.zeros(max(1, B * cols), dtype=np.int32)
    check(lib().pkv_token_table_to_page_table(_ptr(tt), B, W, _ptr(sl), page_size, _ptr(out), out.size))
    return out[: B * cols].reshape(B, cols)
