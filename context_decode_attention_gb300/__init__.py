"""DCP decode attention on one GB300 (sm_103a): thin Python binding of libdcp.

The binding only marshals arguments: every step of the path runs in the CUDA
kernels of libdcp.so (context_decode_attention_gb300/_build/, built by
build.py).  PyTorch supplies device memory and streams.  Nothing here falls
back to the CPU: if the library is missing or cannot load, every call raises.

Functions carry the C ABI's names (include/dcp.h):
  dcp_workspace_size, dcp_workspace_init, dcp_get_error, dcp_slot_mapping, dcp_transfer_blocks, dcp_pcp_partition, dcp_prefill_attention,
  dcp_sparse_workspace_size, dcp_sparse_localize, dcp_sparse_decode_attention,
  dcp_partial_attention, dcp_lse_merge, dcp_decode_attention, dcp_decode_plan, dcp_decode_attention_planned,
  dcp_decode_attention_noalloc,
  dcp_noalloc_get_error
"""

import ctypes
import math
import os

from ._lib import (
    DCP_BF16, DCP_F32, DCP_FP8_E4M3, DCP_LAYOUT_GQA, DCP_LAYOUT_MLA, DcpError, DcpParams, lib, lib_path,
)

__all__ = [
    "DcpError", "DcpParams", "params_from_config", "lib", "lib_path",
    "dcp_workspace_size", "dcp_workspace_init", "dcp_get_error", "dcp_slot_mapping", "dcp_transfer_blocks", "dcp_pcp_partition",
    "dcp_prefill_attention", "dcp_sparse_workspace_size", "dcp_sparse_localize", "dcp_sparse_decode_attention",
    "dcp_partial_attention", "dcp_lse_merge", "dcp_decode_attention", "dcp_decode_plan",
    "dcp_decode_attention_planned", "dcp_decode_attention_noalloc",
    "dcp_noalloc_get_error", "dcp_launch_count",
    "dcp_attention_kernel", "DCP_F32", "DCP_BF16", "DCP_FP8_E4M3", "DCP_LAYOUT_GQA", "DCP_LAYOUT_MLA",
]

_DT = {"f32": DCP_F32, "bf16": DCP_BF16, "fp8": DCP_FP8_E4M3}


def params_from_config(cfg, kv_scale=1.0):
    """dcp_params for a config dict (see dcp_workloads.configs)."""
    p = DcpParams()
    p.N, p.I, p.block_size = int(cfg["N"]), int(cfg["I"]), int(cfg["block_size"])
    p.layout = DCP_LAYOUT_MLA if cfg["layout"] == "mla" else DCP_LAYOUT_GQA
    p.Hq, p.Hkv, p.Dk, p.Dv, p.Tq = (int(cfg[k]) for k in ("Hq", "Hkv", "Dk", "Dv", "Tq"))
    p.q_dtype, p.kv_dtype, p.out_dtype = _DT[cfg["q_dtype"]], _DT[cfg["kv_dtype"]], _DT[cfg["out_dtype"]]
    p.kv_scale = float(kv_scale)
    p.softmax_scale = float(cfg["softmax_scale"])
    return p


def _ptr(t):
    """Device address of a tensor argument.  The library reads and writes
    through plain pointers, so a host tensor or a strided view would be read
    as something else: both are refused here, before any call."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"libdcp takes device tensors; got one on {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"libdcp takes contiguous tensors; got strides {tuple(t.stride())} for shape {tuple(t.shape)}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(rc, what):
    if rc != 0:
        msg = lib().dcp_error_string(rc).decode()
        raise DcpError(rc, f"{what}: {msg} ({rc})")


def dcp_launch_count():
    """Kernel launches libdcp has enqueued since load."""
    return int(lib().dcp_launch_count())


def dcp_attention_kernel(params):
    """Name of the attention kernel libdcp selects for params (None if unsupported)."""
    name = lib().dcp_attention_kernel(ctypes.byref(params))
    return None if name is None else name.decode()


def dcp_workspace_size(params, B, max_seq_len):
    n = ctypes.c_size_t(0)
    _check(lib().dcp_workspace_size(ctypes.byref(params), int(B), int(max_seq_len), ctypes.byref(n)),
           "dcp_workspace_size")
    return int(n.value)


def dcp_workspace_init(workspace, stream=None):
    _check(lib().dcp_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _stream(stream)), "dcp_workspace_init")


def dcp_get_error(workspace, stream=None):
    bits = ctypes.c_uint32(0)
    _check(lib().dcp_get_error(_ptr(workspace), _stream(stream), ctypes.byref(bits)), "dcp_get_error")
    return int(bits.value)


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


# Bytes per element of each dcp_dtype.
_ESIZE = {DCP_F32: 4, DCP_BF16: 2, DCP_FP8_E4M3: 1}


def _need(t, name, nbytes, itemsize):
    """Refuse a buffer with the wrong element size or fewer bytes than the call
    reads or writes through it: the library sees only the address, so a short
    buffer would be read past its end on the device."""
    if t is None:
        return
    if t.element_size() != itemsize:
        raise ValueError(f"{name}: expected {itemsize}-byte elements, got {t.dtype}")
    have = t.numel() * t.element_size()
    if have < nbytes:
        raise ValueError(f"{name}: has {have} bytes; these params and sizes need {nbytes}")


def _kv_row(params):
    """Key and value elements per token row of the pools: (GQA) Hkv x D, (MLA) Dk and none."""
    if params.layout == DCP_LAYOUT_MLA:
        return params.Dk, 0
    return params.Hkv * params.Dk, params.Hkv * params.Dv


def _need_pools(params, k_pool, v_pool, num_blocks):
    kv = _ESIZE.get(params.kv_dtype, 1)
    row_k, row_v = _kv_row(params)
    slots = int(num_blocks) * params.block_size
    _need(k_pool, "k_pool", slots * row_k * kv, kv)
    if row_v:
        _need(v_pool, "v_pool", slots * row_v * kv, kv)


def _need_attention(params, B, q, k_pool, v_pool, num_blocks, block_tables, seq_lens, local_lens):
    """Sizes of the inputs every attention entry point reads (layouts in include/dcp.h)."""
    rows = B * params.Tq * params.Hq
    _need(q, "q", rows * params.Dk * _ESIZE.get(params.q_dtype, 1), _ESIZE.get(params.q_dtype, 1))
    _need_pools(params, k_pool, v_pool, num_blocks)
    _need(block_tables, "block_tables", params.N * B * int(block_tables.shape[-1]) * 4, 4)
    _need(seq_lens, "seq_lens", B * 4, 4)
    _need(local_lens, "local_lens", params.N * B * 4, 4)
    return rows


def dcp_slot_mapping(params, seq_lens, tok_req=None, tok_pos=None, block_tables=None, num_blocks=0,
                     owner=None, slots=None, local_lens=None, virt_blocks=None, rank_blocks=None,
                     new_k=None, new_v=None, k_pool=None, v_pool=None, workspace=None, stream=None):
    B = int(seq_lens.numel())
    T = 0 if tok_req is None else int(tok_req.numel())
    max_blocks = 0 if block_tables is None else int(block_tables.shape[-1])
    N = params.N
    _need(seq_lens, "seq_lens", B * 4, 4)
    _need(tok_req, "tok_req", T * 4, 4)
    _need(tok_pos, "tok_pos", T * 8, 8)
    _need(block_tables, "block_tables", N * B * max_blocks * 4, 4)
    _need(owner, "owner", T, 1)
    _need(slots, "slots", N * T * 8, 8)
    _need(local_lens, "local_lens", N * B * 4, 4)
    _need(virt_blocks, "virt_blocks", B * 4, 4)
    _need(rank_blocks, "rank_blocks", N * B * 4, 4)
    kv = _ESIZE.get(params.kv_dtype, 1)
    row_k, row_v = _kv_row(params)
    _need(new_k, "new_k", T * row_k * kv, kv)
    _need(new_v, "new_v", T * row_v * kv, kv)
    _need_pools(params, k_pool, v_pool, num_blocks)
    _check(lib().dcp_slot_mapping(ctypes.byref(params), B, _ptr(seq_lens), T, _ptr(tok_req), _ptr(tok_pos),
                                  _ptr(block_tables), max_blocks, int(num_blocks), _ptr(owner), _ptr(slots),
                                  _ptr(local_lens), _ptr(virt_blocks), _ptr(rank_blocks), _ptr(new_k),
                                  _ptr(new_v), _ptr(k_pool), _ptr(v_pool), _ptr(workspace),
                                  _nbytes(workspace), _stream(stream)), "dcp_slot_mapping")


def dcp_transfer_blocks(params, seq_lens, block_tables, num_blocks, counts, blocks=None, fills=None,
                        totals=None, workspace=None, stream=None):
    """Per-rank non-empty blocks of each request with their token counts (and
    the batch's slots / tokens moved in totals[2]); see include/dcp.h."""
    B, M, N = int(seq_lens.numel()), int(block_tables.shape[-1]), params.N
    _need(seq_lens, "seq_lens", B * 4, 4)
    _need(block_tables, "block_tables", N * B * M * 4, 4)
    _need(counts, "counts", N * B * 4, 4)
    _need(blocks, "blocks", N * B * M * 4, 4)
    _need(fills, "fills", N * B * M * 4, 4)
    _need(totals, "totals", 2 * 8, 8)
    _check(lib().dcp_transfer_blocks(ctypes.byref(params), int(seq_lens.numel()), _ptr(seq_lens),
                                     _ptr(block_tables), int(block_tables.shape[-1]), int(num_blocks),
                                     _ptr(counts), _ptr(blocks), _ptr(fills), _ptr(totals), _ptr(workspace),
                                     _nbytes(workspace), _stream(stream)), "dcp_transfer_blocks")


def dcp_pcp_partition(K, ctx_lens, q_lens, max_q, pos, padded_lens, workspace=None, stream=None):
    """Head-tail prefill partition over K PCP ranks into pos [B, max_q] (gathered
    order, -1 = padding) and padded_lens [B]; see include/dcp.h."""
    B = int(ctx_lens.numel())
    _need(ctx_lens, "ctx_lens", B * 4, 4)
    _need(q_lens, "q_lens", B * 4, 4)
    _need(pos, "pos", B * max(0, int(max_q)) * 4, 4)
    _need(padded_lens, "padded_lens", B * 4, 4)
    _check(lib().dcp_pcp_partition(int(K), int(ctx_lens.numel()), _ptr(ctx_lens), _ptr(q_lens), int(max_q),
                                   _ptr(pos), _ptr(padded_lens), _ptr(workspace), _nbytes(workspace),
                                   _stream(stream)), "dcp_pcp_partition")


def dcp_prefill_attention(params, q, q_pos, k_pool, v_pool, num_blocks, block_tables, seq_lens, local_lens,
                          out_partial, lse_partial, out=None, lse=None, workspace=None, stream=None):
    """Causal prefill of gathered query rows q [B, Tq, Hq, D] at positions
    q_pos [B, Tq]: per-rank partials, and the merged output when `out` is
    given; see include/dcp.h."""
    B, Tq, N = int(q.shape[0]), int(q.shape[1]), params.N
    rows = B * Tq * params.Hq
    qs, os_ = _ESIZE.get(params.q_dtype, 1), _ESIZE.get(params.out_dtype, 1)
    _need(q, "q", rows * params.Dk * qs, qs)
    _need(q_pos, "q_pos", B * Tq * 4, 4)
    _need_pools(params, k_pool, v_pool, num_blocks)
    _need(block_tables, "block_tables", N * B * int(block_tables.shape[-1]) * 4, 4)
    _need(seq_lens, "seq_lens", B * 4, 4)
    _need(local_lens, "local_lens", N * B * 4, 4)
    _need(out_partial, "out_partial", N * rows * params.Dv * 4, 4)
    _need(lse_partial, "lse_partial", N * rows * 4, 4)
    _need(out, "out", rows * params.Dv * os_, os_)
    _need(lse, "lse", rows * 4, 4)
    _check(lib().dcp_prefill_attention(ctypes.byref(params), int(q.shape[0]), int(q.shape[1]), _ptr(q), _ptr(q_pos),
                                       _ptr(k_pool), _ptr(v_pool), int(num_blocks), _ptr(block_tables),
                                       int(block_tables.shape[-1]), _ptr(seq_lens), _ptr(local_lens),
                                       _ptr(out_partial), _ptr(lse_partial), _ptr(out), _ptr(lse), _ptr(workspace),
                                       _nbytes(workspace), _stream(stream)), "dcp_prefill_attention")


def dcp_sparse_workspace_size(params, B, k):
    n = ctypes.c_size_t(0)
    _check(lib().dcp_sparse_workspace_size(ctypes.byref(params), int(B), int(k), ctypes.byref(n)),
           "dcp_sparse_workspace_size")
    return int(n.value)


def dcp_sparse_localize(params, cand, seq_lens, local, counts, workspace=None, stream=None):
    """Each rank's candidates (cand [B*Tq, k]) at their local positions; see include/dcp.h."""
    R, k, N = int(seq_lens.numel()) * params.Tq, int(cand.shape[-1]), params.N
    _need(cand, "cand", R * k * 4, 4)
    _need(seq_lens, "seq_lens", int(seq_lens.numel()) * 4, 4)
    _need(local, "local", N * R * k * 4, 4)
    _need(counts, "counts", N * R * 4, 4)
    _check(lib().dcp_sparse_localize(ctypes.byref(params), int(seq_lens.numel()), int(cand.shape[-1]), _ptr(cand),
                                     _ptr(seq_lens), _ptr(local), _ptr(counts), _ptr(workspace), _nbytes(workspace),
                                     _stream(stream)), "dcp_sparse_localize")


def dcp_sparse_decode_attention(params, q, cand, k_pool, num_blocks, block_tables, seq_lens, out, lse=None,
                                workspace=None, stream=None):
    """Attention of every query row over its candidate positions only, DCP-localised; see include/dcp.h."""
    B, k, N = int(q.shape[0]), int(cand.shape[-1]), params.N
    rows = B * params.Tq * params.Hq
    qs, os_ = _ESIZE.get(params.q_dtype, 1), _ESIZE.get(params.out_dtype, 1)
    _need(q, "q", rows * params.Dk * qs, qs)
    _need(cand, "cand", B * params.Tq * k * 4, 4)
    _need_pools(params, k_pool, None, num_blocks)
    _need(block_tables, "block_tables", N * B * int(block_tables.shape[-1]) * 4, 4)
    _need(seq_lens, "seq_lens", B * 4, 4)
    _need(out, "out", rows * params.Dv * os_, os_)
    _need(lse, "lse", rows * 4, 4)
    _check(lib().dcp_sparse_decode_attention(ctypes.byref(params), int(q.shape[0]), int(cand.shape[-1]), _ptr(q),
                                             _ptr(cand), _ptr(k_pool), int(num_blocks), _ptr(block_tables),
                                             int(block_tables.shape[-1]), _ptr(seq_lens), _ptr(out), _ptr(lse),
                                             _ptr(workspace), _nbytes(workspace), _stream(stream)),
           "dcp_sparse_decode_attention")


def dcp_partial_attention(params, q, k_pool, v_pool, num_blocks, block_tables, seq_lens, local_lens,
                          out_partial, lse_partial, workspace, stream=None):
    B = int(seq_lens.numel())
    rows = _need_attention(params, B, q, k_pool, v_pool, num_blocks, block_tables, seq_lens, local_lens)
    _need(out_partial, "out_partial", params.N * rows * params.Dv * 4, 4)
    _need(lse_partial, "lse_partial", params.N * rows * 4, 4)
    _check(lib().dcp_partial_attention(ctypes.byref(params), int(seq_lens.numel()), _ptr(q), _ptr(k_pool),
                                       _ptr(v_pool), int(num_blocks), _ptr(block_tables),
                                       int(block_tables.shape[-1]), _ptr(seq_lens), _ptr(local_lens),
                                       _ptr(out_partial), _ptr(lse_partial), _ptr(workspace),
                                       _nbytes(workspace), _stream(stream)), "dcp_partial_attention")


def _need_decode_out(params, rows, out, lse):
    _need(out, "out", rows * params.Dv * _ESIZE.get(params.out_dtype, 1), _ESIZE.get(params.out_dtype, 1))
    _need(lse, "lse", rows * 4, 4)


def dcp_decode_attention(params, q, k_pool, v_pool, num_blocks, block_tables, seq_lens, local_lens,
                         out, lse, workspace, stream=None):
    B = int(seq_lens.numel())
    rows = _need_attention(params, B, q, k_pool, v_pool, num_blocks, block_tables, seq_lens, local_lens)
    _need_decode_out(params, rows, out, lse)
    _check(lib().dcp_decode_attention(ctypes.byref(params), int(seq_lens.numel()), _ptr(q), _ptr(k_pool),
                                      _ptr(v_pool), int(num_blocks), _ptr(block_tables),
                                      int(block_tables.shape[-1]), _ptr(seq_lens), _ptr(local_lens),
                                      _ptr(out), _ptr(lse), _ptr(workspace), _nbytes(workspace),
                                      _stream(stream)), "dcp_decode_attention")


def dcp_decode_plan(params, seq_lens, local_lens, max_blocks, workspace, stream=None):
    """The work plan of dcp_decode_attention_planned, made ahead (include/dcp.h):
    it depends on the lengths only, so it can run beside the step's cache write
    or once for every layer of a step."""
    B = int(seq_lens.numel())
    _need(seq_lens, "seq_lens", B * 4, 4)
    _need(local_lens, "local_lens", params.N * B * 4, 4)
    _check(lib().dcp_decode_plan(ctypes.byref(params), B, _ptr(seq_lens), _ptr(local_lens), int(max_blocks),
                                 _ptr(workspace), _nbytes(workspace), _stream(stream)), "dcp_decode_plan")


def dcp_decode_attention_planned(params, q, k_pool, v_pool, num_blocks, block_tables, seq_lens, local_lens,
                                 out, lse, workspace, stream=None):
    """dcp_decode_attention on the plan dcp_decode_plan left in the workspace
    (same arguments; a plan for other arguments raises DCP_DEV_ERR_PLAN)."""
    B = int(seq_lens.numel())
    rows = _need_attention(params, B, q, k_pool, v_pool, num_blocks, block_tables, seq_lens, local_lens)
    _need_decode_out(params, rows, out, lse)
    _check(lib().dcp_decode_attention_planned(ctypes.byref(params), B, _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                              int(num_blocks), _ptr(block_tables), int(block_tables.shape[-1]),
                                              _ptr(seq_lens), _ptr(local_lens), _ptr(out), _ptr(lse),
                                              _ptr(workspace), _nbytes(workspace), _stream(stream)),
           "dcp_decode_attention_planned")


def dcp_lse_merge(N, rows, Dv, out_partial, lse_partial, out, out_dtype, lse=None, stream=None):
    n = max(0, int(N)) * max(0, int(rows))
    _need(out_partial, "out_partial", n * int(Dv) * 4, 4)
    _need(lse_partial, "lse_partial", n * 4, 4)
    _need(out, "out", max(0, int(rows)) * int(Dv) * _ESIZE.get(int(out_dtype), 1), _ESIZE.get(int(out_dtype), 1))
    _need(lse, "lse", max(0, int(rows)) * 4, 4)
    _check(lib().dcp_lse_merge(int(N), int(rows), int(Dv), _ptr(out_partial), _ptr(lse_partial), _ptr(out),
                               int(out_dtype), _ptr(lse), _stream(stream)), "dcp_lse_merge")


def dcp_decode_attention_noalloc(params, q, k_pool, v_pool, num_blocks, block_tables, seq_lens, local_lens,
                                 out, lse, stream=None):
    """dcp_decode_attention on the library's static scratch (no workspace argument).

    For callers that cannot allocate device memory (a plugin in an engine that
    owns all device memory, or a path that cannot afford an allocation's
    latency or failure).  Calls must not overlap on the GPU: they share one
    scratch buffer.  See include/dcp.h.
    """
    B = int(seq_lens.numel())
    rows = _need_attention(params, B, q, k_pool, v_pool, num_blocks, block_tables, seq_lens, local_lens)
    _need_decode_out(params, rows, out, lse)
    _check(lib().dcp_decode_attention_noalloc(ctypes.byref(params), int(seq_lens.numel()), _ptr(q), _ptr(k_pool),
                                              _ptr(v_pool), int(num_blocks), _ptr(block_tables),
                                              int(block_tables.shape[-1]), _ptr(seq_lens), _ptr(local_lens),
                                              _ptr(out), _ptr(lse), _stream(stream)),
           "dcp_decode_attention_noalloc")


def dcp_noalloc_get_error(stream=None):
    """Device error bits the last dcp_decode_attention_noalloc call on this
    device left in the library's static buffer (read and cleared; waits for
    the stream).  Allocates nothing."""
    bits = ctypes.c_uint32(0)
    _check(lib().dcp_noalloc_get_error(_stream(stream), ctypes.byref(bits)), "dcp_noalloc_get_error")
    return int(bits.value)
