"""Torch-facing wrappers with the C ABI's names.

Argument marshalling only: shapes and dtypes are read off the tensors, outputs
and the workspace are allocated with torch when the caller passes none, and the
call is enqueued on torch's current CUDA stream.  All computation happens in
libspecverify.so.
"""

from __future__ import annotations

import contextlib
import ctypes

import torch

from . import _lib
from ._lib import SpecParams

_DT = {torch.float32: _lib.SPEC_F32, torch.bfloat16: _lib.SPEC_BF16}
_KIND = {"logits": _lib.SPEC_DRAFT_LOGITS, "probs": _lib.SPEC_DRAFT_PROBS}


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensors are required")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _dt(t):
    if t is None:
        return _lib.SPEC_F32
    if t.dtype not in _DT:
        raise ValueError(f"unsupported dtype {t.dtype}")
    return _DT[t.dtype]


def _want(t, dtype, shape, name):
    """Dtype and shape check of an argument (the C ABI sees only pointers)."""
    if t.dtype != dtype or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be {dtype} of shape {tuple(shape)}, "
                         f"got {t.dtype} {tuple(t.shape)}")


def _stream(stream):
    """The caller's stream, else torch's current stream of the current
    device (the wrappers make the tensors' device current first)."""
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _device(primary, *others, stream=None):
    """The device of `primary`.  Every other tensor given (inputs, outputs,
    workspace) and the stream must be on it: the library launches on the
    current device and would otherwise touch another GPU's memory."""
    dev = primary.device
    for t in others:
        if t is not None and t.device != dev:
            raise ValueError(f"all tensors must be on {dev}; got one on "
                             f"{t.device}")
    if stream is not None and dev.type == "cuda" and stream.device != dev:
        raise ValueError(f"stream is on {stream.device}, tensors on {dev}")
    return dev


def _on(dev):
    """Make `dev` the current CUDA device for the call (launch device and
    current stream follow it)."""
    if dev.type == "cuda":
        return torch.cuda.device(dev)
    return contextlib.nullcontext()  # host-side tests with CPU tensors


def params(temperature=1.0, top_k=0, top_p=1.0, draft_kind="logits", seed=0,
           offset=0, draft_lse=None, flags=0) -> SpecParams:
    if draft_lse is not None:
        if draft_lse.dtype != torch.float32 or not draft_lse.is_contiguous():
            raise ValueError("draft_lse must be a contiguous float32 tensor")
    return SpecParams(float(temperature), int(top_k), float(top_p),
                      _KIND[draft_kind], int(seed) & (2**64 - 1),
                      int(offset) & 0xFFFFFFFF, int(flags) & 0xFFFFFFFF,
                      None if draft_lse is None else draft_lse.data_ptr())


def spec_workspace_bytes(op: int, B: int, n: int, V: int) -> int:
    return int(_lib.call("spec_workspace_bytes", op, B, n, V))


def workspace(op, B, n, V, device=None):
    nbytes = spec_workspace_bytes(op, B, n, V)
    if nbytes == 0:
        raise ValueError("invalid sizes for the workspace")
    return torch.empty(nbytes, dtype=torch.uint8,
                       device=device or torch.cuda.current_device())


def spec_verify_chain(target, draft, draft_tokens, *, temperature=1.0,
                      top_k=0, top_p=1.0, draft_kind="logits", seed=0,
                      offset=0, out=None, ws=None, stream=None):
    """target [B, K+1, V]; draft [B, K, V] (None at temperature 0);
    draft_tokens [B, K] int32.  Returns (accepted [B], tokens [B, K+1],
    accept_mass [B, K])."""
    B, K1, V = target.shape
    K = K1 - 1
    dev = target.device
    if out is None:
        out = (torch.empty(B, dtype=torch.int32, device=dev),
               torch.empty(B, K + 1, dtype=torch.int32, device=dev),
               torch.empty(B, K, dtype=torch.float32, device=dev))
    _want(out[0], torch.int32, (B,), "accepted")
    _want(out[1], torch.int32, (B, K + 1), "tokens")
    _want(out[2], torch.float32, (B, K), "accept_mass")
    if ws is None:
        ws = workspace(_lib.SPEC_OP_CHAIN, B, K, V, dev)
    _device(target, draft, draft_tokens, *out, ws, stream=stream)
    prm = params(temperature, top_k, top_p, draft_kind, seed, offset)
    with _on(dev):
        _lib.call("spec_verify_chain", _ptr(target), _ptr(draft),
                  _ptr(draft_tokens), B, K, V, _dt(target), _dt(draft),
                  ctypes.byref(prm), _ptr(out[0]), _ptr(out[1]),
                  _ptr(out[2]), _ptr(ws), ws.numel(), _stream(stream))
    return out


def spec_verify_tree(target, draft, q_row, node_tokens, parent, *,
                     temperature=1.0, top_k=0, top_p=1.0, draft_kind="logits",
                     seed=0, offset=0, out=None, ws=None, stream=None,
                     draft_lse=None):
    """target [B, N+1, V]; draft [B, R, V]; q_row [B, N+1]; node_tokens and
    parent [B, N]; draft_lse [B, R] float32 (optional): the draft rows' log2
    normalisers at this temperature, as spec_eagle2_expand_rerank writes
    them.  Returns (path_len [B], path_nodes [B, N], tokens [B, N+1],
    accept_mass [B, N+1])."""
    B, N1, V = target.shape
    N = N1 - 1
    R = 0 if draft is None else draft.shape[1]
    dev = target.device
    if out is None:
        out = (torch.empty(B, dtype=torch.int32, device=dev),
               torch.empty(B, N, dtype=torch.int32, device=dev),
               torch.empty(B, N + 1, dtype=torch.int32, device=dev),
               torch.empty(B, N + 1, dtype=torch.float32, device=dev))
    _want(out[0], torch.int32, (B,), "path_len")
    _want(out[1], torch.int32, (B, N), "path_nodes")
    _want(out[2], torch.int32, (B, N + 1), "tokens")
    _want(out[3], torch.float32, (B, N + 1), "accept_mass")
    if ws is None:
        ws = workspace(_lib.SPEC_OP_TREE, B, N, V, dev)
    _device(target, draft, q_row, node_tokens, parent, draft_lse, *out, ws,
            stream=stream)
    prm = params(temperature, top_k, top_p, draft_kind, seed, offset,
                 draft_lse)
    with _on(dev):
        _lib.call("spec_verify_tree", _ptr(target), _ptr(draft), _ptr(q_row),
                  _ptr(node_tokens), _ptr(parent), B, N, R, V, _dt(target),
                  _dt(draft), ctypes.byref(prm), _ptr(out[0]), _ptr(out[1]),
                  _ptr(out[2]), _ptr(out[3]), _ptr(ws), ws.numel(),
                  _stream(stream))
    return out


def spec_lm_head(hidden, w_vocab, *, temperature=0.0, row_lse=False,
                 out=None, ws=None, stream=None):
    """Target logits = hidden [..., H] x w_vocab^T (w_vocab [V, H]), bf16.
    Returns (logits [..., V] bf16, row_lse [...] float32 or None): with
    row_lse=True (temperature > 0) also each row's base-2 log normaliser
    log2 sum_v 2^(z_v log2(e) / temperature), taken in the GEMM epilogue."""
    H = hidden.shape[-1]
    V = w_vocab.shape[0]
    lead = tuple(hidden.shape[:-1])
    M = 1
    for d in lead:
        M *= d
    _want(hidden, torch.bfloat16, lead + (H,), "hidden")
    _want(w_vocab, torch.bfloat16, (V, H), "w_vocab")
    dev = hidden.device
    if out is None:
        out = torch.empty(lead + (V,), dtype=torch.bfloat16, device=dev)
    _want(out, torch.bfloat16, lead + (V,), "logits")
    lse = (torch.empty(lead, dtype=torch.float32, device=dev)
           if row_lse else None)
    if ws is None:
        ws = workspace(_lib.SPEC_OP_LMHEAD, M, 0, V, dev)
    _device(hidden, w_vocab, out, lse, ws, stream=stream)
    with _on(dev):
        _lib.call("spec_lm_head", _ptr(hidden), _ptr(w_vocab), M, H, V,
                  float(temperature), _ptr(out), _ptr(lse), _ptr(ws),
                  ws.numel(), _stream(stream))
    return out, lse


def spec_verify_tree_lmhead(hidden, w_vocab, draft, q_row, node_tokens,
                            parent, *, temperature=1.0, top_k=0, top_p=1.0,
                            draft_kind="logits", seed=0, offset=0,
                            logits=None, out=None, ws=None, stream=None,
                            draft_lse=None, flags=0):
    """Tree verification whose target logits are hidden [B, N+1, H] x
    w_vocab^T (bf16; see spec_verify_tree for the rest).  logits: an
    optional [B, N+1, V] bf16 tensor that receives the computed logits.
    Returns (path_len, path_nodes, tokens, accept_mass)."""
    B, N1, H = hidden.shape
    N = N1 - 1
    V = w_vocab.shape[0]
    R = 0 if draft is None else draft.shape[1]
    dev = hidden.device
    _want(hidden, torch.bfloat16, (B, N1, H), "hidden")
    _want(w_vocab, torch.bfloat16, (V, H), "w_vocab")
    if logits is not None:
        _want(logits, torch.bfloat16, (B, N1, V), "logits")
    if out is None:
        out = (torch.empty(B, dtype=torch.int32, device=dev),
               torch.empty(B, N, dtype=torch.int32, device=dev),
               torch.empty(B, N + 1, dtype=torch.int32, device=dev),
               torch.empty(B, N + 1, dtype=torch.float32, device=dev))
    _want(out[0], torch.int32, (B,), "path_len")
    _want(out[1], torch.int32, (B, N), "path_nodes")
    _want(out[2], torch.int32, (B, N + 1), "tokens")
    _want(out[3], torch.float32, (B, N + 1), "accept_mass")
    if ws is None:
        ws = workspace(_lib.SPEC_OP_TREE_LMHEAD, B, N, V, dev)
    _device(hidden, w_vocab, draft, q_row, node_tokens, parent, logits,
            draft_lse, *out, ws, stream=stream)
    prm = params(temperature, top_k, top_p, draft_kind, seed, offset,
                 draft_lse, flags)
    with _on(dev):
        _lib.call("spec_verify_tree_lmhead", _ptr(hidden), _ptr(w_vocab), H,
                  _ptr(draft), _ptr(q_row), _ptr(node_tokens), _ptr(parent),
                  B, N, R, V, _dt(draft), ctypes.byref(prm), _ptr(out[0]),
                  _ptr(out[1]), _ptr(out[2]), _ptr(out[3]), _ptr(logits),
                  _ptr(ws), ws.numel(), _stream(stream))
    return out


def spec_tree_mask(parent, *, bits=False, mask=True, stream=None):
    """parent [B, N] int32 -> (mask [B, N, N] uint8 or None,
    bits [B, N] int64 (uint64 bit patterns) or None)."""
    B, N = parent.shape
    dev = _device(parent, stream=stream)
    m = torch.empty(B, N, N, dtype=torch.uint8, device=dev) if mask else None
    bt = torch.empty(B, N, dtype=torch.int64, device=dev) if bits else None
    with _on(dev):
        _lib.call("spec_tree_mask", _ptr(parent), B, N, _ptr(m), _ptr(bt),
                  _stream(stream))
    return m, bt


def spec_eagle2_expand_rerank(draft_logits, *, temperature, depth=6, topk=10,
                              width=10, total=60, mask=True, out=None,
                              ws=None, stream=None, draft_lse=None):
    """draft_logits [B, 1 + (depth-1)*width, V].  Returns (node_tokens,
    parent, q_row, value, mask).  draft_lse [B, R] float32 (optional) is
    filled with each draft row's log2 normaliser, for spec_verify_tree."""
    B, R, V = draft_logits.shape
    dev = draft_logits.device
    if out is None:
        out = (torch.empty(B, total, dtype=torch.int32, device=dev),
               torch.empty(B, total, dtype=torch.int32, device=dev),
               torch.empty(B, total + 1, dtype=torch.int32, device=dev),
               torch.empty(B, total, dtype=torch.float32, device=dev),
               torch.empty(B, total, total, dtype=torch.uint8, device=dev)
               if mask else None)
    if ws is None:
        ws = workspace(_lib.SPEC_OP_EAGLE2, B, R, V, dev)
    _want(out[0], torch.int32, (B, total), "node_tokens")
    _want(out[1], torch.int32, (B, total), "parent")
    _want(out[2], torch.int32, (B, total + 1), "q_row")
    _want(out[3], torch.float32, (B, total), "value")
    if out[4] is not None:
        _want(out[4], torch.uint8, (B, total, total), "mask")
    if draft_lse is not None and tuple(draft_lse.shape) != (B, R):
        raise ValueError("draft_lse must have shape [B, R]")
    _device(draft_logits, *out, ws, draft_lse, stream=stream)
    prm = params(temperature, draft_lse=draft_lse)
    with _on(dev):
        _lib.call("spec_eagle2_expand_rerank", _ptr(draft_logits), B, V,
                  _dt(draft_logits), depth, topk, width, total,
                  ctypes.byref(prm), _ptr(out[0]), _ptr(out[1]),
                  _ptr(out[2]), _ptr(out[3]), _ptr(out[4]), _ptr(ws),
                  ws.numel(), _stream(stream))
    return out


def spec_kv_commit(kv, prefix_len, path_len, path_nodes=None, *, layout,
                   row_bytes, N, new_len=None, stream=None):
    """Keep the accepted drafts' KV entries (see the C declaration).
    kv: the cache tensor (its storage is addressed in bytes); layout: the
    byte strides (n1, n2, stride_b, stride_1, stride_2, stride_pos);
    prefix_len, path_len [B] int32; path_nodes [B, N] int32 or None (chain).
    Returns new_len [B] int32."""
    B = prefix_len.numel()
    if new_len is None:
        new_len = torch.empty(B, dtype=torch.int32, device=prefix_len.device)
    _want(new_len, torch.int32, (B,), "new_len")
    dev = _device(kv, prefix_len, path_len, path_nodes, new_len,
                  stream=stream)
    n1, n2, sb, s1, s2, sp = layout
    with _on(dev):
        _lib.call("spec_kv_commit", _ptr(kv), B, n1, n2, sb, s1, s2, sp,
                  row_bytes, _ptr(prefix_len), _ptr(path_nodes),
                  _ptr(path_len), N, _ptr(new_len), _stream(stream))
    return new_len


def accept_stats_records(n, nbins=20, device=None):
    """Zeroed records for spec_accept_stats (a dict of device tensors)."""
    dev = device or torch.cuda.current_device()
    z = lambda k, dt=torch.int64: torch.zeros(k, dtype=dt, device=dev)
    return {"len_hist": z(n + 1), "node_tested": z(n), "node_accepted": z(n),
            "depth_tested": z(n), "depth_accepted": z(n),
            "calib_tested": z(nbins), "calib_accepted": z(nbins),
            "calib_conf_sum": z(nbins, torch.float64), "invalid": z(1)}


def spec_accept_stats(count, parent=None, path_nodes=None, confidence=None,
                      *, n, nbins=20, out=None, stream=None):
    """Add one batch of verification outcomes to the acceptance records.
    count [B] int32 (chain accepted counts or tree path_len); parent and
    path_nodes [B, n] int32 for a tree (None for a chain); confidence [B, n]
    float32 or None.  out: the records (accept_stats_records), added to and
    returned; entries may be None to skip them."""
    B = count.numel()
    _want(count, torch.int32, (B,), "count")
    if (parent is None) != (path_nodes is None):
        raise ValueError("parent and path_nodes go together (tree) or are "
                         "both None (chain)")
    if parent is not None:
        _want(parent, torch.int32, (B, n), "parent")
        _want(path_nodes, torch.int32, (B, n), "path_nodes")
    if confidence is not None:
        _want(confidence, torch.float32, (B, n), "confidence")
    if out is None:
        out = accept_stats_records(n, nbins, count.device)
    sizes = {"len_hist": n + 1, "node_tested": n, "node_accepted": n,
             "depth_tested": n, "depth_accepted": n, "calib_tested": nbins,
             "calib_accepted": nbins, "calib_conf_sum": nbins, "invalid": 1}
    for f, k in sizes.items():  # the kernel writes int64 / float64 records
        if out.get(f) is not None:
            _want(out[f], torch.float64 if f == "calib_conf_sum"
                  else torch.int64, (k,), f)
    dev = _device(count, parent, path_nodes, confidence,
                  *[out.get(f) for f in _lib.STATS_FIELDS], stream=stream)
    rec = _lib.SpecAcceptStats(*[
        None if out.get(f) is None else _ptr(out[f]).value
        for f in _lib.STATS_FIELDS])
    with _on(dev):
        _lib.call("spec_accept_stats", _ptr(count), _ptr(parent),
                  _ptr(path_nodes), _ptr(confidence), B, n, nbins,
                  ctypes.byref(rec), _stream(stream))
    return out


def spec_tree_attention(q, k_cache, v_cache, prefix_len, mask_bits, *,
                        scale=None, out=None, stream=None):
    """q [B, N, Hq, D] bf16; k_cache, v_cache [B, Hkv, S, D] bf16;
    prefix_len [B] int32; mask_bits [B, N] int64 (uint64 bit patterns from
    spec_tree_mask).  Returns out [B, N, Hq, D] bf16."""
    B, N, Hq, D = q.shape
    _, Hkv, S, _ = k_cache.shape
    _want(q, torch.bfloat16, (B, N, Hq, D), "q")
    _want(k_cache, torch.bfloat16, (B, Hkv, S, D), "k_cache")
    _want(v_cache, torch.bfloat16, (B, Hkv, S, D), "v_cache")
    _want(prefix_len, torch.int32, (B,), "prefix_len")
    _want(mask_bits, torch.int64, (B, N), "mask_bits")
    if out is None:
        out = torch.empty_like(q)
    _want(out, torch.bfloat16, (B, N, Hq, D), "out")
    if scale is None:
        scale = D ** -0.5
    dev = _device(q, k_cache, v_cache, prefix_len, mask_bits, out,
                  stream=stream)
    with _on(dev):
        _lib.call("spec_tree_attention", _ptr(q), _ptr(k_cache),
                  _ptr(v_cache), _ptr(prefix_len), _ptr(mask_bits), B, N, Hq,
                  Hkv, D, S, float(scale), _ptr(out), _stream(stream))
    return out


def spec_get_status(ws, stream=None) -> int:
    v = ctypes.c_uint32(0)
    with _on(_device(ws, stream=stream)):
        _lib.call("spec_get_status", _ptr(ws), ctypes.byref(v),
                  _stream(stream))
    return int(v.value)


def spec_philox_uniforms(seed, offset, b, idx, slot, stream=None):
    n = b.numel()
    dev = _device(b, idx, slot, stream=stream)
    out = torch.empty(n, dtype=torch.float32, device=dev)
    with _on(dev):
        _lib.call("spec_philox_uniforms", int(seed) & (2**64 - 1),
                  int(offset) & 0xFFFFFFFF, _ptr(b), _ptr(idx), _ptr(slot), n,
                  _ptr(out), _stream(stream))
    return out
