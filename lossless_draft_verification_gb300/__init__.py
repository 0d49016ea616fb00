"""Python binding of the specv C ABI (lossless draft verification on GB300).

Two layers, both argument marshalling only (every step of the computation runs
in the CUDA library ``_lib/libspecv.so``):

* ``specv_*`` -- one function per C entry point with the same name and
  argument order; pointers are passed as integers (``tensor.data_ptr()``) and
  the return value is the integer ``specv_status``.
* ``verify_chain``, ``tv_accept``, ``verify_tree_greedy``, ``markov_draft``,
  ``schedule`` -- tensor-level helpers: they check dtype/shape/device,
  allocate outputs and the workspace with torch on the tensors' device, call
  the C entry point on the current torch stream and raise ``SpecvError`` on a
  non-zero status.  ``verify_chain`` also accepts host tensors: inputs are
  copied to the device and the results back (the end-to-end path).

There is no fallback: if the shared library is missing, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "load", "SpecvError", "SPECV_OK", "SPECV_ERR_INVALID_ARG", "SPECV_ERR_UNSUPPORTED", "SPECV_ERR_CUDA",
    "SPECV_ERR_DEVICE_DATA", "SPECV_ERR_TIMEOUT", "SPECV_ERR_SCRATCH_LIMIT", "SPECV_F32", "SPECV_BF16", "EXPORTED",
    "specv_verify_chain_workspace_size", "specv_verify_chain", "specv_verify_chain_noalloc", "specv_tv_accept_workspace_size", "specv_tv_accept",
    "specv_verify_tree_greedy_workspace_size", "specv_verify_tree_greedy", "specv_markov_draft_workspace_size",
    "specv_markov_draft", "specv_markov_recompute_logits_workspace_size", "specv_markov_recompute_logits",
    "specv_schedule_workspace_size", "specv_schedule", "specv_schedule_global", "specv_prune_threshold",
    "specv_confidence_head_workspace_size", "specv_confidence_head", "specv_dart_tree_workspace_size",
    "specv_dart_tree",
    "specv_read_device_error", "specv_selftest_bounded_wait",
    "specv_status_string", "specv_abi_version", "specv_shard_combine_normalisers", "specv_shard_pick",
    "specv_shard_argmax_combine",
    "verify_chain", "tv_accept", "verify_tree_greedy", "markov_draft", "markov_recompute_logits", "schedule",
    "schedule_global",
    "prune_threshold", "confidence_head", "dart_tree", "read_device_error",
]

(SPECV_OK, SPECV_ERR_INVALID_ARG, SPECV_ERR_UNSUPPORTED, SPECV_ERR_CUDA, SPECV_ERR_DEVICE_DATA, SPECV_ERR_TIMEOUT,
 SPECV_ERR_SCRATCH_LIMIT) = range(7)
SPECV_F32, SPECV_BF16 = 0, 1

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libspecv.so")

_c_int, _c_size, _c_float, _c_double, _vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_float, ctypes.c_double, ctypes.c_void_p

# name -> (restype, argtypes); every symbol declared in include/specv.h
EXPORTED = {
    "specv_verify_chain_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "specv_verify_chain": (_c_int, [_vp, _vp, _c_int, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_float, _vp, _vp, _vp,
                                    _vp, _c_size, _vp]),
    "specv_verify_chain_noalloc": (_c_int, [_vp, _vp, _c_int, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_float, _vp, _vp,
                                            _vp, _vp]),
    "specv_tv_accept_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "specv_tv_accept": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_float, _vp, _vp, _c_size, _vp]),
    "specv_verify_tree_greedy_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "specv_verify_tree_greedy": (_c_int, [_vp, _c_int, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _vp, _vp,
                                          _c_size, _vp]),
    "specv_markov_draft_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "specv_markov_draft": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_float, _vp, _vp,
                                    _c_int, _vp, _c_size, _vp]),
    "specv_markov_recompute_logits_workspace_size": (_c_size, [_c_int, _c_int]),
    "specv_markov_recompute_logits": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _vp, _vp,
                                               _c_size, _vp]),
    "specv_schedule_workspace_size": (_c_size, [_c_int, _c_int]),
    "specv_schedule": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _vp, _vp, _vp, _c_size, _vp]),
    "specv_schedule_global": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_int, _vp, _vp, _vp, _c_size, _vp]),
    "specv_prune_threshold": (_c_int, [_vp, _c_int, _c_int, _c_double, _vp, _vp, _c_size, _vp]),
    "specv_confidence_head_workspace_size": (_c_size, [_c_int, _c_int]),
    "specv_dart_tree_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "specv_dart_tree": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_float, _c_int, _c_int, _c_int, _vp, _vp, _vp,
                                 _vp, _c_size, _vp]),
    "specv_confidence_head": (_c_int, [_vp, _vp, _vp, _c_float, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp,
                                       _vp, _c_size, _vp]),
    "specv_read_device_error": (_c_int, [_vp, _vp, ctypes.POINTER(ctypes.c_int32)]),
    "specv_selftest_bounded_wait": (_c_int, [ctypes.c_uint32, _c_int, _vp, _c_size, _vp]),
    "specv_status_string": (ctypes.c_char_p, [_c_int]),
    "specv_abi_version": (_c_int, []),
    "specv_shard_combine_normalisers": (_c_int, [_vp, _c_int, _c_int, _vp]),
    "specv_shard_pick": (_c_int, [_vp, _c_int, _c_int, _vp, _vp, _vp]),
    "specv_shard_argmax_combine": (_c_int, [_vp, _vp, _c_int, _c_int, _vp]),
}

_lib = None


class SpecvError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} (status {status})")
        self.status = status


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libspecv.so (built by lossless_draft_verification_gb300.build)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise FileNotFoundError(f"{p} is missing: build it with `python -m lossless_draft_verification_gb300.build`")
    lib = ctypes.CDLL(p)
    for name, (res, args) in EXPORTED.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().specv_status_string(status).decode()


def _call(name, *args):
    return getattr(load(), name)(*args)


# --------------------------------------------------------------------------- raw entry points
def specv_verify_chain_workspace_size(R, gamma, V, dtype):
    return _call("specv_verify_chain_workspace_size", R, gamma, V, dtype)


def specv_verify_chain(target_logits, draft_logits, dtype, draft_tokens, lengths, uniforms, R, gamma, V, temperature,
                       accepted_len, out_token, c_star, workspace, workspace_bytes, stream):
    return _call("specv_verify_chain", target_logits, draft_logits, dtype, draft_tokens, lengths, uniforms, R, gamma,
                 V, temperature, accepted_len, out_token, c_star, workspace, workspace_bytes, stream)


def specv_verify_chain_noalloc(target_logits, draft_logits, dtype, draft_tokens, lengths, uniforms, R, gamma, V,
                               temperature, accepted_len, out_token, c_star, stream):
    return _call("specv_verify_chain_noalloc", target_logits, draft_logits, dtype, draft_tokens, lengths, uniforms, R,
                 gamma, V, temperature, accepted_len, out_token, c_star, stream)


def specv_tv_accept_workspace_size(R, gamma, V, dtype):
    return _call("specv_tv_accept_workspace_size", R, gamma, V, dtype)


def specv_tv_accept(target_logits, draft_logits, dtype, R, gamma, target_positions, V, temperature, c_star, workspace,
                    workspace_bytes, stream):
    return _call("specv_tv_accept", target_logits, draft_logits, dtype, R, gamma, target_positions, V, temperature,
                 c_star, workspace, workspace_bytes, stream)


def specv_verify_tree_greedy_workspace_size(R, N, V, dtype):
    return _call("specv_verify_tree_greedy_workspace_size", R, N, V, dtype)


def specv_verify_tree_greedy(target_logits, dtype, parents, tokens, R, N, V, max_depth, path_len, path_nodes,
                             out_token, workspace, workspace_bytes, stream):
    return _call("specv_verify_tree_greedy", target_logits, dtype, parents, tokens, R, N, V, max_depth, path_len,
                 path_nodes, out_token, workspace, workspace_bytes, stream)


def specv_markov_draft_workspace_size(R, gamma, V, rank):
    return _call("specv_markov_draft_workspace_size", R, gamma, V, rank)


def specv_markov_draft(U, W1, W2, anchor, uniforms, R, gamma, V, rank, temperature, draft_tokens, draft_logits,
                       logits_out_dtype, workspace, workspace_bytes, stream):
    return _call("specv_markov_draft", U, W1, W2, anchor, uniforms, R, gamma, V, rank, temperature, draft_tokens,
                 draft_logits, logits_out_dtype, workspace, workspace_bytes, stream)


def specv_markov_recompute_logits_workspace_size(R, gamma):
    return _call("specv_markov_recompute_logits_workspace_size", R, gamma)


def specv_markov_recompute_logits(U, W1, W2, anchor, draft_tokens, lengths, R, gamma, V, rank, draft_logits, workspace,
                                  workspace_bytes, stream):
    return _call("specv_markov_recompute_logits", U, W1, W2, anchor, draft_tokens, lengths, R, gamma, V, rank,
                 draft_logits, workspace, workspace_bytes, stream)


def specv_schedule_workspace_size(R, gamma):
    return _call("specv_schedule_workspace_size", R, gamma)


def specv_schedule(conf, sps, R, gamma, B_max, lengths, theta_best, workspace, workspace_bytes, stream):
    return _call("specv_schedule", conf, sps, R, gamma, B_max, lengths, theta_best, workspace, workspace_bytes, stream)


def specv_schedule_global(conf, conf_stale, sps, R, gamma, B_max, lengths, theta_best, workspace, workspace_bytes,
                          stream):
    return _call("specv_schedule_global", conf, conf_stale, sps, R, gamma, B_max, lengths, theta_best, workspace,
                 workspace_bytes, stream)


def specv_prune_threshold(conf, R, gamma, threshold, lengths, workspace, workspace_bytes, stream):
    return _call("specv_prune_threshold", conf, R, gamma, threshold, lengths, workspace, workspace_bytes, stream)


def specv_confidence_head_workspace_size(R, gamma):
    return _call("specv_confidence_head_workspace_size", R, gamma)


def specv_confidence_head(h, W1, w, b, anchor, draft_tokens, R, gamma, H, V, rank, conf, workspace, workspace_bytes,
                          stream):
    return _call("specv_confidence_head", h, W1, w, b, anchor, draft_tokens, R, gamma, H, V, rank, conf, workspace,
                 workspace_bytes, stream)


def specv_dart_tree_workspace_size(R, d, V, k, w, theta, dtype):
    return _call("specv_dart_tree_workspace_size", R, d, V, k, w, theta, dtype)


def specv_dart_tree(draft_logits, dtype, R, d, V, temperature, k, w, theta, parents, tokens, n_nodes, workspace,
                    workspace_bytes, stream):
    return _call("specv_dart_tree", draft_logits, dtype, R, d, V, temperature, k, w, theta, parents, tokens, n_nodes,
                 workspace, workspace_bytes, stream)


def specv_read_device_error(workspace, stream, status_out):
    return _call("specv_read_device_error", workspace, stream, status_out)


def specv_selftest_bounded_wait(max_polls, arrive, workspace, workspace_bytes, stream):
    return _call("specv_selftest_bounded_wait", max_polls, arrive, workspace, workspace_bytes, stream)


def specv_status_string(status):
    return _call("specv_status_string", status)


def specv_abi_version():
    return _call("specv_abi_version")


# host arrays (e.g. numpy ``.ctypes.data`` or CPU tensors' ``data_ptr()``)
def specv_shard_combine_normalisers(part, shards, rows, out):
    return _call("specv_shard_combine_normalisers", part, shards, rows, out)


def specv_shard_pick(mass, shards, rows, u, shard_out, target_out):
    return _call("specv_shard_pick", mass, shards, rows, u, shard_out, target_out)


def specv_shard_argmax_combine(val, idx, shards, rows, out):
    return _call("specv_shard_argmax_combine", val, idx, shards, rows, out)


# --------------------------------------------------------------------------- tensor helpers
def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return SPECV_BF16
    if t.dtype == torch.float32:
        return SPECV_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _p(t) -> int | None:
    return None if t is None else t.data_ptr()


def _check(t, name, device, dtype=None, shape=None):
    if t is None:
        return
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _stream_ptr(stream) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _workspace(nbytes: int, device, workspace=None):
    torch = _torch()
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small")
        return workspace
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def _raise(status, where):
    if status != SPECV_OK:
        raise SpecvError(status, where)


_copy_streams = {}


def _copy_streams_for(dev):
    """Two copy streams per device, created once (stream creation is not free)."""
    torch = _torch()
    key = dev.index
    if key not in _copy_streams:
        _copy_streams[key] = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    return _copy_streams[key]


def _verify_chain_host_chunked(target, draft, draft_tokens, uniforms, temperature, lengths, want_c_star, chunks,
                               stream):
    """Host inputs, requests split into `chunks` groups: group i's host-to-device
    copies run on copy stream i % 2 while the verification of group i - 1 runs
    on the compute stream, so the copies overlap the kernels (and the two copy
    streams can use two copy engines)."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device())
    comp = stream if stream is not None else torch.cuda.current_stream(dev)
    R, P, V = target.shape
    gamma = P - 1
    nb = target.is_pinned()
    d_t = torch.empty(target.shape, dtype=target.dtype, device=dev)
    d_d = None if draft is None else torch.empty(draft.shape, dtype=draft.dtype, device=dev)
    d_x = torch.empty(draft_tokens.shape, dtype=draft_tokens.dtype, device=dev)
    d_u = None if uniforms is None else torch.empty(uniforms.shape, dtype=uniforms.dtype, device=dev)
    d_l = None if lengths is None else torch.empty(lengths.shape, dtype=lengths.dtype, device=dev)
    # the three outputs share one device buffer, so one transfer returns them
    out = torch.empty(2 * R + (R * gamma if want_c_star else 0), dtype=torch.int32, device=dev)
    acc, tok = out[:R], out[R:2 * R]
    cst = out[2 * R:].view(torch.float32).view(R, gamma) if want_c_star else None
    code = _dtype_code(target)
    copies = _copy_streams_for(dev)
    for c in copies:
        c.wait_stream(comp)                 # the device buffers were allocated on the compute stream
    step = -(-R // chunks)
    ws = None
    for i, r0 in enumerate(range(0, R, step)):
        r1 = min(R, r0 + step)
        cs = copies[i % 2]
        with torch.cuda.stream(cs):
            for d, h in ((d_t, target), (d_d, draft), (d_x, draft_tokens), (d_u, uniforms), (d_l, lengths)):
                if d is not None:
                    d[r0:r1].copy_(h[r0:r1], non_blocking=nb)
        ev = torch.cuda.Event()
        ev.record(cs)
        comp.wait_event(ev)
        n = r1 - r0
        nbytes = specv_verify_chain_workspace_size(n, gamma, V, code)
        if nbytes == 0:
            raise SpecvError(SPECV_ERR_UNSUPPORTED, "specv_verify_chain_workspace_size")
        if ws is None:
            ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        sl = lambda t: None if t is None else t[r0:r1]
        st = specv_verify_chain(_p(sl(d_t)), _p(sl(d_d)), code, _p(sl(d_x)), _p(sl(d_l)), _p(sl(d_u)), n, gamma, V,
                                float(temperature), _p(sl(acc)), _p(sl(tok)), _p(sl(cst)), _p(ws), ws.numel(),
                                comp.cuda_stream)
        _raise(st, "specv_verify_chain")
    for t in (d_t, d_d, d_x, d_u, d_l):
        if t is not None:
            for c in copies:
                t.record_stream(c)
    with torch.cuda.stream(comp):
        h = out.cpu()
    return h[:R], h[R:2 * R], (h[2 * R:].view(torch.float32).view(R, gamma) if want_c_star else None)


def verify_chain(target, draft, draft_tokens, uniforms, temperature: float, lengths=None, want_c_star: bool = True,
                 workspace=None, stream=None, out=None, chunks: int = 1):
    """Chain speculative sampling (see specv_verify_chain in include/specv.h).

    target [R, gamma+1, V], draft [R, gamma, V] (bf16 or float32), draft_tokens
    [R, gamma] int32, uniforms [R, gamma+1, 2] float32 (None at T = 0), lengths
    [R] int32 or None.  Returns (accepted_len [R], out_token [R], c_star [R, gamma]
    or None) on the inputs' device.  Host (CPU) inputs are copied to the current
    CUDA device first and the results copied back; with chunks > 1 the requests
    go in that many groups whose copies overlap the previous group's kernels
    (pinned host tensors make the copies asynchronous)."""
    torch = _torch()
    host = target.device.type == "cpu"
    if host and chunks > 1 and out is None and workspace is None and target.shape[0] > 1:
        return _verify_chain_host_chunked(target, draft, draft_tokens, uniforms, temperature, lengths, want_c_star,
                                          min(int(chunks), target.shape[0]), stream)
    if host:
        dev = torch.device("cuda", torch.cuda.current_device())
        nb = target.is_pinned()
        target = target.to(dev, non_blocking=nb)
        draft = None if draft is None else draft.to(dev, non_blocking=nb)
        draft_tokens = draft_tokens.to(dev, non_blocking=nb)
        uniforms = None if uniforms is None else uniforms.to(dev, non_blocking=nb)
        lengths = None if lengths is None else lengths.to(dev, non_blocking=nb)
    R, P, V = target.shape
    gamma = P - 1
    dev = target.device
    _check(target, "target", dev)
    _check(draft, "draft", dev, target.dtype, (R, gamma, V))
    _check(draft_tokens, "draft_tokens", dev, torch.int32, (R, gamma))
    _check(uniforms, "uniforms", dev, torch.float32, (R, gamma + 1, 2))
    _check(lengths, "lengths", dev, torch.int32, (R,))
    code = _dtype_code(target)
    if out is None:
        acc = torch.empty(R, dtype=torch.int32, device=dev)
        tok = torch.empty(R, dtype=torch.int32, device=dev)
        cst = torch.empty(R, gamma, dtype=torch.float32, device=dev) if want_c_star else None
    else:
        acc, tok, cst = out
    nbytes = specv_verify_chain_workspace_size(R, gamma, V, code)
    if nbytes == 0:
        raise SpecvError(SPECV_ERR_UNSUPPORTED, "specv_verify_chain_workspace_size")
    ws = _workspace(nbytes, dev, workspace)
    st = specv_verify_chain(_p(target), _p(draft), code, _p(draft_tokens), _p(lengths), _p(uniforms), R, gamma, V,
                            float(temperature), _p(acc), _p(tok), _p(cst), _p(ws), ws.numel(), _stream_ptr(stream))
    _raise(st, "specv_verify_chain")
    if host:
        return acc.cpu(), tok.cpu(), None if cst is None else cst.cpu()
    return acc, tok, cst


def tv_accept(target, draft, temperature: float, workspace=None, stream=None):
    """c*_{r,k} = 1 - 1/2 ||p_k - q_k||_1 for target [R, P >= gamma, V], draft [R, gamma, V]."""
    torch = _torch()
    R, P, V = target.shape
    gamma = draft.shape[1]
    dev = target.device
    _check(target, "target", dev)
    _check(draft, "draft", dev, target.dtype, (R, gamma, V))
    code = _dtype_code(target)
    cst = torch.empty(R, gamma, dtype=torch.float32, device=dev)
    nbytes = specv_tv_accept_workspace_size(R, gamma, V, code)
    if nbytes == 0:
        raise SpecvError(SPECV_ERR_UNSUPPORTED, "specv_tv_accept_workspace_size")
    ws = _workspace(nbytes, dev, workspace)
    st = specv_tv_accept(_p(target), _p(draft), code, R, gamma, P, V, float(temperature), _p(cst), _p(ws), ws.numel(),
                         _stream_ptr(stream))
    _raise(st, "specv_tv_accept")
    return cst


def verify_tree_greedy(target, parents, tokens, max_depth: int, workspace=None, stream=None):
    """Greedy tree verification; target [R, N+1, V], parents/tokens [R, N+1] int32.
    Returns (path_len [R], path_nodes [R, max_depth], out_token [R])."""
    torch = _torch()
    R, N1, V = target.shape
    dev = target.device
    _check(target, "target", dev)
    _check(parents, "parents", dev, torch.int32, (R, N1))
    _check(tokens, "tokens", dev, torch.int32, (R, N1))
    code = _dtype_code(target)
    plen = torch.empty(R, dtype=torch.int32, device=dev)
    nodes = torch.empty(R, max_depth, dtype=torch.int32, device=dev)
    tok = torch.empty(R, dtype=torch.int32, device=dev)
    nbytes = specv_verify_tree_greedy_workspace_size(R, N1 - 1, V, code)
    if nbytes == 0:
        raise SpecvError(SPECV_ERR_UNSUPPORTED, "specv_verify_tree_greedy_workspace_size")
    ws = _workspace(nbytes, dev, workspace)
    st = specv_verify_tree_greedy(_p(target), code, _p(parents), _p(tokens), R, N1 - 1, V, int(max_depth), _p(plen),
                                  _p(nodes), _p(tok), _p(ws), ws.numel(), _stream_ptr(stream))
    _raise(st, "specv_verify_tree_greedy")
    return plen, nodes, tok


def markov_draft(U, W1, W2, anchor, uniforms, temperature: float, want_logits: bool = True, logits_dtype=None,
                 workspace=None, stream=None):
    """Markov-head drafting; U [R, gamma, V], W1 [V, rank], W2 [rank, V] bf16, anchor [R]
    int32, uniforms [R, gamma] float32.  Returns (draft_tokens [R, gamma], logits or None)."""
    torch = _torch()
    R, gamma, V = U.shape
    rank = W1.shape[1]
    dev = U.device
    _check(U, "U", dev, torch.bfloat16)
    _check(W1, "W1", dev, torch.bfloat16, (V, rank))
    _check(W2, "W2", dev, torch.bfloat16, (rank, V))
    _check(anchor, "anchor", dev, torch.int32, (R,))
    _check(uniforms, "uniforms", dev, torch.float32, (R, gamma))
    toks = torch.empty(R, gamma, dtype=torch.int32, device=dev)
    ldt = logits_dtype or torch.float32
    logits = torch.empty(R, gamma, V, dtype=ldt, device=dev) if want_logits else None
    code = SPECV_BF16 if ldt == torch.bfloat16 else SPECV_F32
    nbytes = specv_markov_draft_workspace_size(R, gamma, V, rank)
    ws = _workspace(nbytes, dev, workspace)
    st = specv_markov_draft(_p(U), _p(W1), _p(W2), _p(anchor), _p(uniforms), R, gamma, V, rank, float(temperature),
                            _p(toks), _p(logits), code, _p(ws), ws.numel(), _stream_ptr(stream))
    _raise(st, "specv_markov_draft")
    return toks, logits


def markov_recompute_logits(U, W1, W2, anchor, draft_tokens, lengths=None, out=None, workspace=None, stream=None):
    """Draft logits of the verified positions (k < lengths[r]) recomputed after
    drafting without kept logits; returns `out` [R, gamma, V] bf16 (other rows
    untouched; a new uninitialised tensor when out is None)."""
    torch = _torch()
    R, gamma, V = U.shape
    rank = W1.shape[1]
    dev = U.device
    _check(U, "U", dev, torch.bfloat16)
    _check(W1, "W1", dev, torch.bfloat16, (V, rank))
    _check(W2, "W2", dev, torch.bfloat16, (rank, V))
    _check(anchor, "anchor", dev, torch.int32, (R,))
    _check(draft_tokens, "draft_tokens", dev, torch.int32, (R, gamma))
    _check(lengths, "lengths", dev, torch.int32, (R,))
    if out is None:
        out = torch.empty(R, gamma, V, dtype=torch.bfloat16, device=dev)
    _check(out, "out", dev, torch.bfloat16, (R, gamma, V))
    nbytes = specv_markov_recompute_logits_workspace_size(R, gamma)
    ws = _workspace(nbytes, dev, workspace)
    st = specv_markov_recompute_logits(_p(U), _p(W1), _p(W2), _p(anchor), _p(draft_tokens), _p(lengths), R, gamma, V,
                                       rank, _p(out), _p(ws), ws.numel(), _stream_ptr(stream))
    _raise(st, "specv_markov_recompute_logits")
    return out


def schedule(conf, sps, B_max: int | None = None, workspace=None, stream=None):
    """Greedy throughput scheduler; conf [R, gamma] float32, sps [B_max] float64.
    Returns (lengths [R] int32, theta_best [1] float64)."""
    torch = _torch()
    R, gamma = conf.shape
    dev = conf.device
    _check(conf, "conf", dev, torch.float32)
    _check(sps, "sps", dev, torch.float64)
    B_max = sps.shape[0] if B_max is None else B_max
    lengths = torch.empty(R, dtype=torch.int32, device=dev)
    theta = torch.empty(1, dtype=torch.float64, device=dev)
    nbytes = specv_schedule_workspace_size(R, gamma)
    ws = _workspace(nbytes, dev, workspace)
    st = specv_schedule(_p(conf), _p(sps), R, gamma, int(B_max), _p(lengths), _p(theta), _p(ws), ws.numel(),
                        _stream_ptr(stream))
    _raise(st, "specv_schedule")
    return lengths, theta


def schedule_global(conf, sps, conf_stale=None, B_max: int | None = None, workspace=None, stream=None):
    """Asynchronous global-search scheduler: the count K from conf_stale (or
    conf when None), no early stop; the entries from conf.  conf and conf_stale
    [R, gamma] float32, sps [B_max] float64.  Returns (lengths [R] int32,
    theta_best [1] float64)."""
    torch = _torch()
    R, gamma = conf.shape
    dev = conf.device
    _check(conf, "conf", dev, torch.float32)
    _check(conf_stale, "conf_stale", dev, torch.float32, (R, gamma))
    _check(sps, "sps", dev, torch.float64)
    B_max = sps.shape[0] if B_max is None else B_max
    lengths = torch.empty(R, dtype=torch.int32, device=dev)
    theta = torch.empty(1, dtype=torch.float64, device=dev)
    nbytes = specv_schedule_workspace_size(R, gamma)
    ws = _workspace(nbytes, dev, workspace)
    st = specv_schedule_global(_p(conf), _p(conf_stale), _p(sps), R, gamma, int(B_max), _p(lengths), _p(theta),
                               _p(ws), ws.numel(), _stream_ptr(stream))
    _raise(st, "specv_schedule_global")
    return lengths, theta


def prune_threshold(conf, threshold: float, workspace=None, stream=None):
    """Confidence-threshold suffix pruning; conf [R, gamma] float32.  Returns
    lengths [R] int32: the leading positions whose running product of
    confidences stays >= threshold."""
    torch = _torch()
    R, gamma = conf.shape
    dev = conf.device
    _check(conf, "conf", dev, torch.float32)
    lengths = torch.empty(R, dtype=torch.int32, device=dev)
    nbytes = specv_schedule_workspace_size(R, gamma)
    ws = _workspace(nbytes, dev, workspace)
    st = specv_prune_threshold(_p(conf), R, gamma, float(threshold), _p(lengths), _p(ws), ws.numel(),
                               _stream_ptr(stream))
    _raise(st, "specv_prune_threshold")
    return lengths


def confidence_head(h, W1, w, b: float, anchor, draft_tokens, workspace=None, stream=None):
    """DSpark's confidence head: h [R, gamma, H] bf16, W1 [V, rank] bf16,
    w [H + rank] float32, anchor [R] and draft_tokens [R, gamma] int32.
    Returns conf [R, gamma] float32."""
    torch = _torch()
    R, gamma, H = h.shape
    V, rank = W1.shape
    dev = h.device
    _check(h, "h", dev, torch.bfloat16)
    _check(W1, "W1", dev, torch.bfloat16)
    _check(w, "w", dev, torch.float32, (H + rank,))
    _check(anchor, "anchor", dev, torch.int32, (R,))
    _check(draft_tokens, "draft_tokens", dev, torch.int32, (R, gamma))
    conf = torch.empty(R, gamma, dtype=torch.float32, device=dev)
    nbytes = specv_confidence_head_workspace_size(R, gamma)
    ws = _workspace(nbytes, dev, workspace)
    st = specv_confidence_head(_p(h), _p(W1), _p(w), float(b), _p(anchor), _p(draft_tokens), R, gamma, H, V, rank,
                               _p(conf), _p(ws), ws.numel(), _stream_ptr(stream))
    _raise(st, "specv_confidence_head")
    return conf


def dart_tree(draft_logits, temperature: float = 1.0, k: int = 25, w: int = 20, theta: int = 59, workspace=None,
              stream=None):
    """DART's candidate tree without the n-gram index; draft_logits [R, d, V]
    bfloat16 or float32.  Returns (parents, tokens [R, theta + 1] int32,
    n_nodes [R] int32): row 0 is the root, rows are in depth-first order."""
    torch = _torch()
    R, d, V = draft_logits.shape
    dev = draft_logits.device
    _check(draft_logits, "draft_logits", dev)
    dt = _dtype_code(draft_logits)
    parents = torch.empty(R, theta + 1, dtype=torch.int32, device=dev)
    tokens = torch.empty(R, theta + 1, dtype=torch.int32, device=dev)
    n_nodes = torch.empty(R, dtype=torch.int32, device=dev)
    nbytes = specv_dart_tree_workspace_size(R, d, V, k, w, theta, dt)
    if nbytes == 0:
        raise SpecvError(SPECV_ERR_UNSUPPORTED, "specv_dart_tree_workspace_size")
    ws = _workspace(nbytes, dev, workspace)
    st = specv_dart_tree(_p(draft_logits), dt, R, d, V, float(temperature), k, w, theta, _p(parents), _p(tokens),
                         _p(n_nodes), _p(ws), ws.numel(), _stream_ptr(stream))
    _raise(st, "specv_dart_tree")
    return parents, tokens, n_nodes


def read_device_error(workspace, stream=None) -> int:
    out = ctypes.c_int32(0)
    st = specv_read_device_error(_p(workspace), _stream_ptr(stream), ctypes.byref(out))
    _raise(st, "specv_read_device_error")
    return out.value
