"""ctypes binding of libpa.so: argument marshalling only.

Every function here derives sizes from torch tensor shapes, passes raw
device pointers and the current CUDA stream to the C ABI of ``include/pa.h``
and raises ``PaError`` on a non-zero status. No arithmetic of the method is
done in Python and there is no fallback: without the compiled library the
calls raise.
"""

import ctypes
import os

import torch

F16, BF16, FP8_E4M3 = 0, 1, 2
DEVERR_SLOT_RANGE = 0x1
DEVERR_BLOCK_RANGE = 0x2
DEVERR_CONTEXT_RANGE = 0x4
DEVERR_TIMEOUT = 0x8
DEVERR_LAYOUT = 0x10
DEVERR_QUERY_START = 0x20
DEVERR_Q_RANGE = 0x40
DEVERR_PREFIX = 0x80

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libpa.so")
_lib = None

_c_int32 = ctypes.c_int32
_c_ptr = ctypes.c_void_p
_c_size = ctypes.c_size_t


class PaError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {status_name(status)}: {last_error_message()}")


def library_path():
    return _LIB_PATH


def lib():
    """The loaded libpa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                               "`python -m paged_kv_cache_288_gb300.build`")
        L = ctypes.CDLL(_LIB_PATH)
        L.pa_version.restype = ctypes.c_int
        L.pa_status_string.restype = ctypes.c_char_p
        L.pa_status_string.argtypes = [ctypes.c_int]
        L.pa_last_error_message.restype = ctypes.c_char_p
        L.pa_kernel_launch_count.restype = ctypes.c_uint64
        L.pa_reshape_and_cache.restype = ctypes.c_int
        L.pa_reshape_and_cache.argtypes = [
            _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int32, _c_int32, _c_int32, _c_int32,
            _c_int32, ctypes.c_int, ctypes.c_int, _c_ptr, _c_ptr, _c_ptr, _c_ptr]
        L.pa_decode.restype = ctypes.c_int
        L.pa_decode.argtypes = [
            _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int32, _c_ptr, _c_int32, _c_int32,
            _c_int32, _c_int32, _c_int32, _c_int32, ctypes.c_float, ctypes.c_int, ctypes.c_int,
            _c_ptr, _c_ptr, _c_int32, _c_int32, _c_ptr, _c_size, _c_ptr, _c_ptr]
        L.pa_decode_workspace_size.restype = _c_size
        L.pa_decode_workspace_size.argtypes = [_c_int32] * 6
        L.pa_decode_split_noalloc.restype = ctypes.c_int
        L.pa_decode_split_noalloc.argtypes = [
            _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int32, _c_ptr, _c_int32, _c_int32,
            _c_int32, _c_int32, _c_int32, _c_int32, ctypes.c_float, ctypes.c_int, ctypes.c_int,
            _c_ptr, _c_ptr, _c_int32, _c_int32, _c_ptr, _c_ptr]
        L.pa_decode_shared_prefix.restype = ctypes.c_int
        L.pa_decode_shared_prefix.argtypes = [
            _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int32, _c_ptr, _c_int32, _c_int32,
            _c_int32, _c_int32, _c_int32, _c_int32, ctypes.c_float, ctypes.c_int, _c_int32,
            _c_ptr, _c_ptr, _c_int32, _c_int32, _c_int32, _c_ptr, _c_size, _c_ptr, _c_ptr]
        L.pa_decode_shared_prefix_workspace_size.restype = _c_size
        L.pa_decode_shared_prefix_workspace_size.argtypes = [_c_int32] * 8
        L.pa_prefill.restype = ctypes.c_int
        L.pa_prefill.argtypes = [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int32, _c_ptr, _c_ptr,
                                 _c_int32, _c_int32, _c_int32, _c_int32, _c_int32, _c_int32,
                                 _c_int32, _c_int32, ctypes.c_float, ctypes.c_int, _c_ptr, _c_ptr]
        L.pa_swap_blocks.restype = ctypes.c_int
        L.pa_swap_blocks.argtypes = [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int32, _c_ptr, _c_int32,
                                     _c_int32, _c_int32, _c_size, _c_ptr, _c_ptr]
        L.pa_copy_blocks.restype = ctypes.c_int
        L.pa_copy_blocks.argtypes = [_c_ptr, _c_ptr, _c_int32, _c_ptr, _c_int32, _c_int32,
                                     _c_size, _c_ptr, _c_ptr]
        _lib = L
    return _lib


def status_name(status):
    return lib().pa_status_string(int(status)).decode()


def last_error_message():
    return lib().pa_last_error_message().decode()


def _dtype_code(t):
    if t == torch.float16:
        return F16
    if t == torch.bfloat16:
        return BF16
    if t in (torch.uint8, torch.float8_e4m3fn):
        return FP8_E4M3
    raise TypeError(f"unsupported dtype {t}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(status, what):
    if status != 0:
        raise PaError(status, what)


def _on_device(what, **tensors):
    """Every given tensor (None is skipped) must be a dense, contiguous CUDA
    tensor on one device: the C ABI takes raw pointers and assumes exactly
    that layout, so a strided view or a host tensor would be misread."""
    device = None
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{what}: {name} must be a CUDA tensor (got {t.device})")
        if not t.is_contiguous():
            raise ValueError(f"{what}: {name} must be contiguous")
        if device is None:
            device = t.device
        elif t.device != device:
            raise ValueError(f"{what}: {name} is on {t.device}, other tensors on {device}")


def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, k_scale=None, v_scale=None,
                      debug_err=None, stream=None):
    """Write new tokens' K/V ([T, Hkv, d]) into the caches ([Nb, Hkv, bs, d]) at their slots."""
    T, Hkv, d = key.shape
    Nb, Hkv2, bs, d2 = k_cache.shape
    if (Hkv, d) != (Hkv2, d2) or value.shape != key.shape or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch between new tokens and caches")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != T:
        raise ValueError("slot_mapping must be int64 [num_tokens]")
    _on_device("reshape_and_cache", key=key, value=value, k_cache=k_cache, v_cache=v_cache,
               slot_mapping=slot_mapping, k_scale=k_scale, v_scale=v_scale, debug_err=debug_err)
    _check(lib().pa_reshape_and_cache(
        _ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), T, Hkv, d, bs,
        Nb, _dtype_code(key.dtype), _dtype_code(k_cache.dtype), _ptr(k_scale), _ptr(v_scale),
        _ptr(debug_err), _stream(stream)), "pa_reshape_and_cache")


def decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, max_context_len,
                          partition_size=0):
    return int(lib().pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                              max_context_len, partition_size))


def decode(out, q, k_cache, v_cache, block_tables, context_lens, scale, max_context_len,
           k_scale=None, v_scale=None, partition_size=0, workspace=None, debug_err=None,
           stream=None):
    """out[B, Hq, d] = paged single-query attention of q[B, Hq, d] over the caches."""
    B, Hq, d = q.shape
    Nb, Hkv, bs, d2 = k_cache.shape
    if d2 != d or out.shape != q.shape or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.numel() != B:
        raise ValueError("block_tables must be [num_seqs, max_blocks]; context_lens [num_seqs]")
    _on_device("decode", out=out, q=q, k_cache=k_cache, v_cache=v_cache, block_tables=block_tables,
               context_lens=context_lens, k_scale=k_scale, v_scale=v_scale, workspace=workspace,
               debug_err=debug_err)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().pa_decode(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), B, Hq, Hkv, d, bs, Nb, float(scale),
        _dtype_code(q.dtype), _dtype_code(k_cache.dtype), _ptr(k_scale), _ptr(v_scale),
        int(max_context_len), int(partition_size), _ptr(workspace), ws_bytes, _ptr(debug_err),
        _stream(stream)), "pa_decode")


def decode_shared_prefix_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                        num_groups, max_group_size, max_prefix_len):
    return int(lib().pa_decode_shared_prefix_workspace_size(
        num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_groups, max_group_size,
        max_prefix_len))


def decode_shared_prefix(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                         max_context_len, group_start, group_prefix, max_group_size,
                         max_prefix_len, workspace, debug_err=None, stream=None):
    """pa_decode for sequences grouped by a shared leading run of blocks.

    group_start (int32 [num_groups + 1]) and group_prefix (int32 [num_groups])
    are device tensors; group g is sequences group_start[g] ..
    group_start[g+1]-1 sharing their first group_prefix[g] tokens. The
    workspace holds decode_shared_prefix_workspace_size() bytes.
    """
    B, Hq, d = q.shape
    Nb, Hkv, bs, d2 = k_cache.shape
    if d2 != d or out.shape != q.shape or v_cache.shape != k_cache.shape or q.dtype != k_cache.dtype:
        raise ValueError("shape or dtype mismatch")
    for t, name in ((block_tables, "block_tables"), (context_lens, "context_lens"),
                    (group_start, "group_start"), (group_prefix, "group_prefix")):
        if t.dtype != torch.int32:
            raise ValueError(f"{name} must be int32")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.numel() != B:
        raise ValueError("block_tables must be [num_seqs, max_blocks]; context_lens [num_seqs]")
    G = group_prefix.numel()
    if group_start.numel() != G + 1:
        raise ValueError("group_start must be [num_groups + 1]")
    _on_device("decode_shared_prefix", out=out, q=q, k_cache=k_cache, v_cache=v_cache,
               block_tables=block_tables, context_lens=context_lens, group_start=group_start,
               group_prefix=group_prefix, workspace=workspace, debug_err=debug_err)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pa_decode_shared_prefix(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), B, Hq, Hkv, d, bs, Nb, float(scale), _dtype_code(q.dtype),
        int(max_context_len), _ptr(group_start), _ptr(group_prefix), G, int(max_group_size),
        int(max_prefix_len), _ptr(workspace), ws_bytes, _ptr(debug_err), _stream(stream)),
        "pa_decode_shared_prefix")


def prefill(out, q, k_cache, v_cache, block_tables, context_lens, query_start, scale,
            max_query_len, debug_err=None, stream=None):
    """out[T, Hq, d] = causal attention of each sequence's chunk of queries (rows
    query_start[i] .. query_start[i+1]-1 of q[T, Hq, d]) over its paged KV."""
    T, Hq, d = q.shape
    Nb, Hkv, bs, d2 = k_cache.shape
    if d2 != d or out.shape != q.shape or v_cache.shape != k_cache.shape or q.dtype != k_cache.dtype:
        raise ValueError("shape or dtype mismatch")
    for t, name in ((block_tables, "block_tables"), (context_lens, "context_lens"),
                    (query_start, "query_start")):
        if t.dtype != torch.int32:
            raise ValueError(f"{name} must be int32")
    B = context_lens.numel()
    if query_start.numel() != B + 1 or block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("query_start must be [num_seqs + 1]; block_tables [num_seqs, width]")
    _on_device("prefill", out=out, q=q, k_cache=k_cache, v_cache=v_cache, block_tables=block_tables,
               context_lens=context_lens, query_start=query_start, debug_err=debug_err)
    _check(lib().pa_prefill(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), _ptr(query_start), B, T, int(max_query_len), Hq, Hkv, d, bs, Nb,
        float(scale), _dtype_code(q.dtype), _ptr(debug_err), _stream(stream)), "pa_prefill")


def decode_split_noalloc(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                         max_context_len, k_scale=None, v_scale=None, partition_size=0,
                         debug_err=None, stream=None):
    """Split-path decode whose partials live in the library's own scratch array.

    For callers that cannot allocate device memory; see pa_decode_split_noalloc
    in include/pa.h for the size limit and the rule that overlapping calls race.
    """
    B, Hq, d = q.shape
    Nb, Hkv, bs, d2 = k_cache.shape
    if d2 != d or out.shape != q.shape or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.numel() != B:
        raise ValueError("block_tables must be [num_seqs, max_blocks]; context_lens [num_seqs]")
    _on_device("decode_split_noalloc", out=out, q=q, k_cache=k_cache, v_cache=v_cache,
               block_tables=block_tables, context_lens=context_lens, k_scale=k_scale,
               v_scale=v_scale, debug_err=debug_err)
    _check(lib().pa_decode_split_noalloc(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), B, Hq, Hkv, d, bs, Nb, float(scale),
        _dtype_code(q.dtype), _dtype_code(k_cache.dtype), _ptr(k_scale), _ptr(v_scale),
        int(max_context_len), int(partition_size), _ptr(debug_err), _stream(stream)),
        "pa_decode_split_noalloc")


def pointer_array(tensors, device):
    """Device int64 array of the tensors' data pointers (for copy_blocks)."""
    return torch.tensor([t.data_ptr() for t in tensors], dtype=torch.int64, device=device)


def copy_blocks(k_ptrs, v_ptrs, block_mapping, num_blocks, block_bytes, debug_err=None,
                stream=None):
    """Copy blocks (src, dst) = block_mapping[p] in every layer; *_ptrs from pointer_array."""
    if block_mapping.dtype != torch.int64 or block_mapping.dim() != 2 or block_mapping.shape[1] != 2:
        raise ValueError("block_mapping must be int64 [num_pairs, 2]")
    if k_ptrs.dtype != torch.int64 or v_ptrs.dtype != torch.int64 or k_ptrs.numel() != v_ptrs.numel():
        raise ValueError("k_ptrs and v_ptrs must be int64 pointer arrays of one entry per layer")
    _on_device("copy_blocks", k_ptrs=k_ptrs, v_ptrs=v_ptrs, block_mapping=block_mapping,
               debug_err=debug_err)
    _check(lib().pa_copy_blocks(
        _ptr(k_ptrs), _ptr(v_ptrs), k_ptrs.numel(), _ptr(block_mapping), block_mapping.shape[0],
        int(num_blocks), int(block_bytes), _ptr(debug_err), _stream(stream)), "pa_copy_blocks")


SWAP_MAX_LAYERS = 64


def _host_ptr_array(tensors):
    arr = (ctypes.c_void_p * max(1, len(tensors)))()
    for i, t in enumerate(tensors):
        arr[i] = t.data_ptr()
    return arr


def swap_blocks(dst_k, dst_v, src_k, src_v, block_mapping, debug_err=None, stream=None):
    """Move blocks (src, dst) = block_mapping[p] from the src pools to the dst pools, K and V,
    in every layer.

    dst_k, dst_v, src_k, src_v are lists (one tensor per layer) of pools shaped
    [num_blocks, ...]; each is a device tensor or a pinned host tensor
    (pin_memory=True). block_mapping is int64 [num_pairs, 2] on the device or
    in pinned host memory.
    """
    n = len(src_k)
    if not (len(src_v) == len(dst_k) == len(dst_v) == n):
        raise ValueError("one K and one V pool per layer on each side")
    if block_mapping.dtype != torch.int64 or block_mapping.dim() != 2 or block_mapping.shape[1] != 2:
        raise ValueError("block_mapping must be int64 [num_pairs, 2]")
    if n == 0:
        return
    blk = src_k[0][0].numel() * src_k[0].element_size()
    for t in list(src_k) + list(src_v) + list(dst_k) + list(dst_v):
        if not t.is_contiguous() or t[0].numel() * t.element_size() != blk:
            raise ValueError("every pool must be contiguous with the same block size")
    src_nb, dst_nb = src_k[0].shape[0], dst_k[0].shape[0]
    if any(t.shape[0] != src_nb for t in src_v) or any(t.shape[0] != dst_nb for t in list(dst_k) + list(dst_v)):
        raise ValueError("the pools of one side must hold the same number of blocks")
    if any(t.shape[0] != src_nb for t in src_k):
        raise ValueError("the pools of one side must hold the same number of blocks")
    _check(lib().pa_swap_blocks(
        _host_ptr_array(dst_k), _host_ptr_array(dst_v), _host_ptr_array(src_k), _host_ptr_array(src_v),
        n, _ptr(block_mapping), block_mapping.shape[0], int(src_nb), int(dst_nb), int(blk),
        _ptr(debug_err), _stream(stream)), "pa_swap_blocks")
