"""ctypes binding of libtreeverify's C ABI (include/treeverify.h).

Argument marshalling only: every step of the path runs in the library's CUDA kernels.
Tensors of one call must be contiguous CUDA tensors on one device; each call is made with
that device current and is enqueued on its current torch stream (it returns at once).
Index inputs (parent, tokens, counts) must be int32 of exactly the shape the kernels
read.  There is no CPU fallback: if the shared library is missing the first call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libtreeverify.so")

TV_F32 = 0
TV_BF16 = 1

TV_DEV_BAD_TREE = 1
TV_DEV_BAD_TOKEN = 2
TV_DEV_TIMEOUT = 4


class TreeVerifyError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed with status {status}: {msg}")
        self.status = status


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t
_U64 = ctypes.c_uint64

_SIGS = {
    "tv_status_string": (ctypes.c_char_p, [_I]),
    "tv_version": (_I, []),
    "tv_selftest_bounded_wait": (_I, [_I, _P, _P]),
    "tv_philox4x32_10": (_I, [_U64, _P, _I, _P, _P]),
    "tv_set_sm_partition": (_I, [_I, _I]),
    "tv_set_attention_variant": (_I, [_I]),
    "tv_set_attention_splits": (_I, [_I]),
    "tv_tree_prep": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
    "tv_prune_tree": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "tv_tree_attention_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "tv_tree_attention_plan": (_I, [_I, _I, _I, _I, _I, _I, _I, _P, _P]),
    "tv_tree_attention": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P, _P]),
    "tv_verify_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "tv_verify_greedy": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "tv_verify_greedy_static": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]),
    "tv_verify_sample": (_I, [_P, _P, _P, _P, _I, _I, _I, _F, _U64, _U64, _I, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "tv_vocab_stats": (_I, [_P, _P, _P, _P, _I, _I, _I, _F, _I, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "tv_commit_accepted_kv": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P]),
    "tv_frontier_topw": (_I, [_P, _P, _I, _I, _I, _P, _P, _P]),
    "tv_expand_workspace_size": (_SZ, [_I, _I, _I]),
    "tv_expand_children": (_I, [_P, _P, _I, _I, _I, _F, _I, _P, _P, _P, _P, _SZ, _P, _P]),
    "tv_select_workspace_size": (_SZ, [_I, _I, _I, _I]),
    "tv_select_subtree": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "tv_select_subtree_adaptive": (_I, [_P, _P, _I, _I, _I, _I, _F, _F, _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
}


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libtreeverify.so (built by ``python -m tree_speculative_decoding_masked_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"libtreeverify.so not found at {_LIB_PATH}; build it with "
                "`python -m tree_speculative_decoding_masked_gb300.build` (needs nvcc 13, sm_103a)")
        lib = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def exported_symbols() -> list:
    return list(_SIGS)


def status_string(status: int) -> str:
    return load_library().tv_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != 0:
        raise TreeVerifyError(fn, status, status_string(status))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return TV_BF16
    if t.dtype == torch.float32:
        return TV_F32
    raise TypeError(f"unsupported dtype {t.dtype}; use torch.bfloat16 or torch.float32")


def _need_cuda(**tensors):
    """Every given tensor is a contiguous CUDA tensor, all on one device; returns that
    device (the call is then made with it current, on its current stream)."""
    dev = None
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{name} is on {t.device}, other arguments on {dev}: one device per call")
    return dev


def _need(name, t, dtype, shape):
    """``t`` has exactly ``dtype`` and ``shape`` (kernels index it by these sizes)."""
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _ndim(name, t, n):
    if len(t.shape) != n:
        raise ValueError(f"{name} must have {n} dimensions, got shape {tuple(t.shape)}")


def _on(dev):
    """Context making ``dev`` the current CUDA device for one library call, so that the
    library's per-device state and torch's current stream are those of the tensors."""
    return torch.cuda.device(dev)


def _workspace(nbytes: int, device, workspace):
    if workspace is not None:
        if not workspace.is_cuda:
            raise ValueError("workspace must be a CUDA tensor")
        if workspace.device != device:
            raise ValueError(f"workspace is on {workspace.device}, the inputs on {device}")
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace smaller than the library's query")
        return workspace
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _out(o, key, shape, dtype, device):
    t = o.get(key)
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    if not t.is_cuda:
        raise ValueError(f"out[{key!r}] must be a CUDA tensor")
    if t.device != device:
        raise ValueError(f"out[{key!r}] is on {t.device}, the inputs on {device}")
    need = shape if isinstance(shape, int) else math.prod(shape)
    if t.dtype != dtype or not t.is_contiguous() or t.numel() < need:
        raise ValueError(f"out[{key!r}] must be a contiguous {dtype} tensor of at least {need} elements")
    return t


def _status_tensor(dev_status, device):
    if dev_status is None:
        return torch.zeros(1, dtype=torch.int32, device=device)
    if not dev_status.is_cuda:
        raise ValueError("dev_status must be a CUDA tensor")
    if dev_status.device != device:
        raise ValueError(f"dev_status is on {dev_status.device}, the inputs on {device}")
    if dev_status.dtype != torch.int32 or dev_status.numel() < 1:
        raise ValueError("dev_status must be an int32 tensor of at least one element")
    return dev_status


def _tree_inputs(parent, tokens, B, N):
    """parent (and tokens) are int32 [B][N]: the kernels read B * N entries of each."""
    _need("parent", parent, torch.int32, (B, N))
    if tokens is not None:
        _need("tokens", tokens, torch.int32, (B, N))


# ------------------------------------------------------------------------------------


def set_sm_partition(verify_sms: int, attention_sms: int):
    """SM shares for running tree_attention and verify_* concurrently (0, 0 = whole device)."""
    _check("tv_set_sm_partition", load_library().tv_set_sm_partition(int(verify_sms), int(attention_sms)))


def philox4x32_10(seed: int, counters):
    """Philox4x32-10 words of counters [n][4] (CUDA int32 tensor, read as uint32) under
    the 64-bit key `seed`: the sampling walk's generator.  Returns [n][4] int32 (bits)."""
    dev = _need_cuda(counters=counters)
    _ndim("counters", counters, 2)
    n = counters.shape[0]
    _need("counters", counters, torch.int32, (n, 4))
    out = torch.empty_like(counters)
    with _on(dev):
        _check("tv_philox4x32_10", load_library().tv_philox4x32_10(
            ctypes.c_uint64(int(seed) & 0xFFFFFFFFFFFFFFFF), _ptr(counters), n, _ptr(out), _stream()))
    return out


def selftest_bounded_wait(wait_us: int, dev_status):
    """Wait on an mbarrier that nothing completes, giving up after wait_us; the kernel
    sets TV_DEV_TIMEOUT in dev_status (a CUDA int32 tensor) and returns."""
    dev = _need_cuda(dev_status=dev_status)
    _status_tensor(dev_status, dev)
    with _on(dev):
        _check("tv_selftest_bounded_wait", load_library().tv_selftest_bounded_wait(int(wait_us), _ptr(dev_status),
                                                                                   _stream()))


def set_attention_variant(variant: int):
    """Tensor-core attention kernel: 0 automatic, 1 one 128-row tile per CTA, 2 paired tiles,
    3 paired tiles with 64-key KV tiles and double-buffered S, 4 variant 3 on a persistent
    grid, 5 variant 3 on SM pairs (M = 256 products over two CTAs; D = 128)."""
    _check("tv_set_attention_variant", load_library().tv_set_attention_variant(int(variant)))


def set_attention_splits(splits: int):
    """KV splits of the tensor-core attention: 0 automatic, 1..8 forced (measurement)."""
    _check("tv_set_attention_splits", load_library().tv_set_attention_splits(int(splits)))


def tree_prep(parent: torch.Tensor, prefix_len: int, *, dev_status=None, out=None):
    """Depth, position ids, packed ancestor mask and child CSR of ``parent`` [B][N]."""
    dev = _need_cuda(parent=parent)
    _ndim("parent", parent, 2)
    B, N = parent.shape
    _tree_inputs(parent, None, B, N)
    lib = load_library()
    W = (N + 31) // 32
    o = out if out is not None else {}
    depth = _out(o, "depth", (B, N), torch.int32, dev)
    pos = _out(o, "pos", (B, N), torch.int32, dev)
    mask = _out(o, "anc_mask", (B, N, W), torch.int32, dev)
    off = _out(o, "child_off", (B, N + 1), torch.int32, dev)
    idx = _out(o, "child_idx", (B, N), torch.int32, dev)
    st = _status_tensor(dev_status, dev)
    with _on(dev):
        _check("tv_tree_prep", lib.tv_tree_prep(_ptr(parent), B, N, int(prefix_len), _ptr(depth), _ptr(pos),
                                                _ptr(mask), _ptr(off), _ptr(idx), _ptr(st), _stream()))
    return {"depth": depth, "pos": pos, "anc_mask": mask, "child_off": off, "child_idx": idx, "dev_status": st}


def prune_tree(parent, conf, max_children: int, depth_limit: int, *, dev_status=None, out=None):
    """PTD width / depth control of parent [B][N] with confidences conf [B][N] float32.
    Returns dict old_to_new, new_parent [B][N], n_kept, new_root [B]."""
    dev = _need_cuda(parent=parent, conf=conf)
    _ndim("parent", parent, 2)
    B, N = parent.shape
    _tree_inputs(parent, None, B, N)
    _need("conf", conf, torch.float32, (B, N))
    lib = load_library()
    o = out if out is not None else {}
    o2n = _out(o, "old_to_new", (B, N), torch.int32, dev)
    npar = _out(o, "new_parent", (B, N), torch.int32, dev)
    nk = _out(o, "n_kept", (B,), torch.int32, dev)
    nr = _out(o, "new_root", (B,), torch.int32, dev)
    st = _status_tensor(dev_status, dev)
    with _on(dev):
        _check("tv_prune_tree", lib.tv_prune_tree(_ptr(parent), _ptr(conf), B, N, int(max_children), int(depth_limit),
                                                  _ptr(o2n), _ptr(npar), _ptr(nk), _ptr(nr), _ptr(st), _stream()))
    return {"old_to_new": o2n, "new_parent": npar, "n_kept": nk, "new_root": nr, "dev_status": st}


def tree_attention_workspace_size(B, Hq, Hkv, D, P, N, dtype) -> int:
    code = TV_BF16 if dtype == torch.bfloat16 else TV_F32
    return int(load_library().tv_tree_attention_workspace_size(B, Hq, Hkv, D, P, N, code))


def tree_attention_plan(B, Hq, Hkv, D, P, N, dtype):
    """(kernel, splits) that tree_attention would launch: kernel 0 CUDA cores, 1 one
    128-row tile per CTA, 2 paired row tiles, 3 paired row tiles with 64-key KV tiles and
    double-buffered S, 4 variant 3 on a persistent grid, 5 variant 3 on SM pairs (tensor
    cores)."""
    code = TV_BF16 if dtype == torch.bfloat16 else TV_F32
    kern, spl = ctypes.c_int(0), ctypes.c_int(0)
    _check("tv_tree_attention_plan", load_library().tv_tree_attention_plan(
        B, Hq, Hkv, D, P, N, code, ctypes.addressof(kern), ctypes.addressof(spl)))
    return kern.value, spl.value


def tree_attention(q, k_cache, v_cache, parent, prefix_len: int, *, scale: float = 0.0, out=None, workspace=None,
                   dev_status=None):
    """Tree-masked GQA attention.  q [B][Hq][N][D]; k_cache, v_cache [B][Hkv][S][D] with
    S >= prefix_len + N; parent int32 [B][N].  workspace: uint8 device tensor of
    tree_attention_workspace_size bytes for the persistent schedule (allocated here when
    omitted; a smaller one runs the paired kernel unsplit)."""
    dev = _need_cuda(q=q, k_cache=k_cache, v_cache=v_cache, parent=parent, out=out)
    _ndim("q", q, 4)
    _ndim("k_cache", k_cache, 4)
    B, Hq, N, D = q.shape
    Hkv, S = k_cache.shape[1], k_cache.shape[2]
    if v_cache.shape != k_cache.shape or k_cache.dtype != q.dtype or v_cache.dtype != q.dtype:
        raise ValueError("k_cache / v_cache must match each other and q's dtype")
    if k_cache.shape[0] != B or k_cache.shape[3] != D:
        raise ValueError(f"k_cache must be [B={B}][Hkv][S][D={D}], got {tuple(k_cache.shape)}")
    if int(prefix_len) < 0 or int(prefix_len) + N > S:
        raise ValueError(f"prefix_len + N must fit the cache rows: {int(prefix_len)} + {N} > {S}")
    _tree_inputs(parent, None, B, N)
    code = _dtype_code(q)
    if out is None:
        out = torch.empty_like(q)
    elif out.dtype != q.dtype or out.shape != q.shape:
        raise ValueError("out must have q's shape and dtype")
    # the workspace is optional here: a smaller one runs the plan that needs none
    ws_need = tree_attention_workspace_size(B, Hq, Hkv, D, prefix_len, N, q.dtype)
    ws = _workspace(0 if workspace is not None else ws_need, dev, workspace)
    st = _status_tensor(dev_status, dev)
    with _on(dev):
        _check("tv_tree_attention",
               load_library().tv_tree_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(parent), B,
                                                Hq, Hkv, D, int(prefix_len), N, S, float(scale), code, _ptr(ws),
                                                ws.numel() * ws.element_size(), _ptr(st), _stream()))
    return out


def commit_accepted_kv(k_cache, v_cache, accepted_nodes, accept_len, prefix_len: int, *, dev_status=None):
    """Move the accepted root path's cache rows P + a_k to P + k, in place, for every KV
    head of k_cache and v_cache [B][Hkv][S][D].  accepted_nodes [B][N], accept_len [B]
    as returned by verify_greedy / verify_sample."""
    dev = _need_cuda(k_cache=k_cache, v_cache=v_cache, accepted_nodes=accepted_nodes, accept_len=accept_len)
    _ndim("k_cache", k_cache, 4)
    _ndim("accepted_nodes", accepted_nodes, 2)
    B, Hkv, S, D = k_cache.shape
    if v_cache.shape != k_cache.shape or v_cache.dtype != k_cache.dtype:
        raise ValueError("k_cache and v_cache must match")
    N = accepted_nodes.shape[1]
    _need("accepted_nodes", accepted_nodes, torch.int32, (B, N))
    _need("accept_len", accept_len, torch.int32, (B,))
    if int(prefix_len) < 0 or int(prefix_len) + N > S:
        raise ValueError(f"prefix_len + N must fit the cache rows: {int(prefix_len)} + {N} > {S}")
    st = _status_tensor(dev_status, dev)
    with _on(dev):
        _check("tv_commit_accepted_kv",
               load_library().tv_commit_accepted_kv(_ptr(k_cache), _ptr(v_cache), _ptr(accepted_nodes),
                                                    _ptr(accept_len), B, Hkv, D, int(prefix_len), N, S,
                                                    _dtype_code(k_cache), _ptr(st), _stream()))
    return k_cache, v_cache


def frontier_topw(scores, count, width: int, *, dev_status=None, out=None):
    """TreeGraft §3.1 frontier: positions of the `width` highest of scores[b][:count[b]]
    (scores [B][C] float32, count [B] int32); ties to the lower position."""
    dev = _need_cuda(scores=scores, count=count, out=out)
    _ndim("scores", scores, 2)
    B, C = scores.shape
    _need("scores", scores, torch.float32, (B, C))
    _need("count", count, torch.int32, (B,))
    if out is None:
        idx = torch.empty(B, width, dtype=torch.int32, device=dev)
    else:
        idx = _out({"idx": out}, "idx", (B, width), torch.int32, dev)
    st = _status_tensor(dev_status, dev)
    with _on(dev):
        _check("tv_frontier_topw", load_library().tv_frontier_topw(_ptr(scores), _ptr(count), B, C, int(width),
                                                                   _ptr(idx), _ptr(st), _stream()))
    return idx


def expand_workspace_size(R, V, m) -> int:
    return int(load_library().tv_expand_workspace_size(R, V, m))


def expand_children(draft_logits, parent_score, m: int, *, temperature: float = 1.0, workspace=None,
                    dev_status=None, out=None):
    """TreeGraft §3.1 children: the top-m tokens of every drafter row [R][V] with their
    probability p and path score s = parent_score * p.  Returns dict token/p/score [R][m]."""
    dev = _need_cuda(draft_logits=draft_logits, parent_score=parent_score)
    _ndim("draft_logits", draft_logits, 2)
    R, V = draft_logits.shape
    _need("parent_score", parent_score, torch.float32, (R,))
    code = _dtype_code(draft_logits)
    o = out if out is not None else {}
    tok = _out(o, "token", (R, m), torch.int32, dev)
    p = _out(o, "p", (R, m), torch.float32, dev)
    sc = _out(o, "score", (R, m), torch.float32, dev)
    ws = _workspace(expand_workspace_size(R, V, m), dev, workspace)
    st = _status_tensor(dev_status, dev)
    with _on(dev):
        _check("tv_expand_children",
               load_library().tv_expand_children(_ptr(draft_logits), _ptr(parent_score), R, V, int(m),
                                                 float(temperature), code, _ptr(tok), _ptr(p), _ptr(sc), _ptr(ws),
                                                 ws.numel() * ws.element_size(), _ptr(st), _stream()))
    return {"token": tok, "p": p, "score": sc, "dev_status": st}


def verify_workspace_size(B, N, V, dtype, sampling: bool) -> int:
    code = TV_BF16 if dtype == torch.bfloat16 else TV_F32
    return int(load_library().tv_verify_workspace_size(B, N, V, code, 1 if sampling else 0))


def _logits_shape(logits):
    _ndim("logits", logits, 3)
    return logits.shape


def verify_greedy(logits, parent, tokens, *, want_stats: bool = False, workspace=None, dev_status=None, out=None):
    """Greedy acceptance.  logits [B][N][V]; parent, tokens int32 [B][N]; returns dict of
    accepted_nodes [B][N], accept_len [B], bonus_token [B], p_draft [B][N] (+ row_lse,
    row_argmax)."""
    dev = _need_cuda(logits=logits, parent=parent, tokens=tokens)
    B, N, V = _logits_shape(logits)
    _tree_inputs(parent, tokens, B, N)
    code = _dtype_code(logits)
    o = out if out is not None else {}
    acc = _out(o, "accepted_nodes", (B, N), torch.int32, dev)
    alen = _out(o, "accept_len", (B), torch.int32, dev)
    bonus = _out(o, "bonus_token", (B), torch.int32, dev)
    pdr = _out(o, "p_draft", (B, N), torch.float32, dev)
    lse = _out(o, "row_lse", (B, N), torch.float32, dev) if want_stats else None
    am = _out(o, "row_argmax", (B, N), torch.int32, dev) if want_stats else None
    ws = _workspace(verify_workspace_size(B, N, V, logits.dtype, False), dev, workspace)
    st = _status_tensor(dev_status, dev)
    with _on(dev):
        _check("tv_verify_greedy",
               load_library().tv_verify_greedy(_ptr(logits), _ptr(parent), _ptr(tokens), B, N, V, code, _ptr(acc),
                                               _ptr(alen), _ptr(bonus), _ptr(pdr), _ptr(lse), _ptr(am), _ptr(ws),
                                               ws.numel() * ws.element_size(), _ptr(st), _stream()))
    res = {"accepted_nodes": acc, "accept_len": alen, "bonus_token": bonus, "p_draft": pdr, "dev_status": st}
    if want_stats:
        res["row_lse"] = lse
        res["row_argmax"] = am
    return res


def verify_greedy_static(logits, parent, tokens, *, want_stats: bool = False, dev_status=None, out=None):
    """Greedy acceptance without a workspace, for callers that cannot allocate device
    memory when they call the library: the scratch lives in a fixed 4 MiB array inside
    the library.  The first call on a device sets that array up (call it once before any
    stream capture); calls that overlap on the GPU race on the shared array.  Same
    results as verify_greedy; problems whose verify_workspace_size(B, N, V, dtype, False)
    exceeds 4 MiB (4194304 bytes) are refused with status TV_ERR_WORKSPACE."""
    dev = _need_cuda(logits=logits, parent=parent, tokens=tokens)
    B, N, V = _logits_shape(logits)
    _tree_inputs(parent, tokens, B, N)
    code = _dtype_code(logits)
    o = out if out is not None else {}
    acc = _out(o, "accepted_nodes", (B, N), torch.int32, dev)
    alen = _out(o, "accept_len", (B), torch.int32, dev)
    bonus = _out(o, "bonus_token", (B), torch.int32, dev)
    pdr = _out(o, "p_draft", (B, N), torch.float32, dev)
    lse = _out(o, "row_lse", (B, N), torch.float32, dev) if want_stats else None
    am = _out(o, "row_argmax", (B, N), torch.int32, dev) if want_stats else None
    st = _status_tensor(dev_status, dev)
    with _on(dev):
        _check("tv_verify_greedy_static",
               load_library().tv_verify_greedy_static(_ptr(logits), _ptr(parent), _ptr(tokens), B, N, V, code,
                                                      _ptr(acc), _ptr(alen), _ptr(bonus), _ptr(pdr), _ptr(lse),
                                                      _ptr(am), _ptr(st), _stream()))
    res = {"accepted_nodes": acc, "accept_len": alen, "bonus_token": bonus, "p_draft": pdr, "dev_status": st}
    if want_stats:
        res["row_lse"] = lse
        res["row_argmax"] = am
    return res


def verify_sample(target_logits, draft_logits, parent, tokens, *, temperature: float, seed: int, round: int,
                  workspace=None, dev_status=None, out=None):
    """Sampling acceptance with residual resampling (Philox4x32-10 draws).  target_logits,
    draft_logits [B][N][V] of one dtype; parent, tokens int32 [B][N]."""
    dev = _need_cuda(target_logits=target_logits, draft_logits=draft_logits, parent=parent, tokens=tokens)
    B, N, V = _logits_shape(target_logits)
    if draft_logits.shape != target_logits.shape or draft_logits.dtype != target_logits.dtype:
        raise ValueError("draft_logits must match target_logits")
    _tree_inputs(parent, tokens, B, N)
    code = _dtype_code(target_logits)
    o = out if out is not None else {}
    acc = _out(o, "accepted_nodes", (B, N), torch.int32, dev)
    alen = _out(o, "accept_len", (B), torch.int32, dev)
    tok = _out(o, "out_token", (B), torch.int32, dev)
    pdr = _out(o, "p_draft", (B, N), torch.float32, dev)
    qdr = _out(o, "q_draft", (B, N), torch.float32, dev)
    ws = _workspace(verify_workspace_size(B, N, V, target_logits.dtype, True), dev, workspace)
    st = _status_tensor(dev_status, dev)
    with _on(dev):
        _check("tv_verify_sample",
               load_library().tv_verify_sample(_ptr(target_logits), _ptr(draft_logits), _ptr(parent), _ptr(tokens),
                                               B, N, V, float(temperature), int(seed) & (2**64 - 1),
                                               int(round) & (2**64 - 1), code, _ptr(acc), _ptr(alen), _ptr(tok),
                                               _ptr(pdr), _ptr(qdr), _ptr(ws), ws.numel() * ws.element_size(),
                                               _ptr(st), _stream()))
    return {"accepted_nodes": acc, "accept_len": alen, "out_token": tok, "p_draft": pdr, "q_draft": qdr,
            "dev_status": st}


def vocab_stats(logits, parent, tokens, *, draft_logits=None, temperature: float = 1.0, workspace=None,
                dev_status=None, out=None):
    """The fused vocab pass alone: per row lse and argmax of logits/T, drafted-token
    probabilities p_draft (and, with draft_logits, draft_row_lse and q_draft).  logits,
    draft_logits [B][N][V]; parent, tokens int32 [B][N]."""
    dev = _need_cuda(logits=logits, draft_logits=draft_logits, parent=parent, tokens=tokens)
    B, N, V = _logits_shape(logits)
    two = draft_logits is not None
    if two and (draft_logits.shape != logits.shape or draft_logits.dtype != logits.dtype):
        raise ValueError("draft_logits must match logits")
    _tree_inputs(parent, tokens, B, N)
    code = _dtype_code(logits)
    o = out if out is not None else {}
    lse = _out(o, "row_lse", (B, N), torch.float32, dev)
    am = _out(o, "row_argmax", (B, N), torch.int32, dev)
    pdr = _out(o, "p_draft", (B, N), torch.float32, dev)
    lse_q = _out(o, "draft_row_lse", (B, N), torch.float32, dev) if two else None
    qdr = _out(o, "q_draft", (B, N), torch.float32, dev) if two else None
    ws = _workspace(verify_workspace_size(B, N, V, logits.dtype, two), dev, workspace)
    st = _status_tensor(dev_status, dev)
    with _on(dev):
        _check("tv_vocab_stats",
               load_library().tv_vocab_stats(_ptr(logits), _ptr(draft_logits), _ptr(parent), _ptr(tokens), B, N, V,
                                             float(temperature), code, _ptr(lse), _ptr(am), _ptr(pdr), _ptr(lse_q),
                                             _ptr(qdr), _ptr(ws), ws.numel() * ws.element_size(), _ptr(st),
                                             _stream()))
    res = {"row_lse": lse, "row_argmax": am, "p_draft": pdr, "dev_status": st}
    if two:
        res["draft_row_lse"] = lse_q
        res["q_draft"] = qdr
    return res


def select_workspace_size(B, d, K, budget) -> int:
    return int(load_library().tv_select_workspace_size(B, d, K, budget))


def select_subtree(marg, pool_tokens, budget: int, root_token, *, dev_status=None, out=None, cost=None):
    """TAPS-style budgeted prefix-closed subtree.  marg [B][d][K] float32 (sorted per
    position), pool_tokens [B][d][K] int32, root_token [B] int32.  With
    cost=(cost_base, cost_per_row) the tree is cut where expected tokens per unit of
    verification cost peak (tv_select_subtree_adaptive)."""
    dev = _need_cuda(marg=marg, pool_tokens=pool_tokens, root_token=root_token)
    if marg.dtype != torch.float32 or pool_tokens.dtype != torch.int32:
        raise TypeError("marg must be float32 and pool_tokens int32")
    _ndim("marg", marg, 3)
    B, d, K = marg.shape
    _need("pool_tokens", pool_tokens, torch.int32, (B, d, K))
    if root_token is not None:
        _need("root_token", root_token, torch.int32, (B,))
    lib = load_library()
    o = out if out is not None else {}
    par = _out(o, "parent", (B, budget), torch.int32, dev)
    tok = _out(o, "tokens", (B, budget), torch.int32, dev)
    dep = _out(o, "depth", (B, budget), torch.int32, dev)
    sc = _out(o, "score", (B, budget), torch.float32, dev)
    nn = _out(o, "n_nodes", (B), torch.int32, dev)
    ws_need = select_workspace_size(B, d, K, budget)
    ws = _workspace(ws_need, dev, None) if ws_need else None
    st = _status_tensor(dev_status, dev)
    with _on(dev):
        if cost is None:
            _check("tv_select_subtree",
                   lib.tv_select_subtree(_ptr(marg), _ptr(pool_tokens), B, d, K, int(budget), _ptr(root_token),
                                         _ptr(par), _ptr(tok), _ptr(dep), _ptr(sc), _ptr(nn), _ptr(ws),
                                         0 if ws is None else ws.numel(), _ptr(st), _stream()))
        else:
            _check("tv_select_subtree_adaptive",
                   lib.tv_select_subtree_adaptive(_ptr(marg), _ptr(pool_tokens), B, d, K, int(budget),
                                                  float(cost[0]), float(cost[1]), _ptr(root_token), _ptr(par),
                                                  _ptr(tok), _ptr(dep), _ptr(sc), _ptr(nn), _ptr(ws),
                                                  0 if ws is None else ws.numel(), _ptr(st), _stream()))
    return {"parent": par, "tokens": tok, "depth": dep, "score": sc, "n_nodes": nn, "dev_status": st}
