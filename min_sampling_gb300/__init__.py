"""Sorting-free top-k / top-p / min-p sampling on GB300 (sm_103a).

Thin Python binding of ``libfs_sampling.so`` (C ABI declared in
``include/fs_sampling.h``).  This module only marshals arguments: it checks
tensor shapes, dtypes and devices, turns scalar parameters into per-row device
arrays, and passes raw device pointers and the current CUDA stream to the library.
Every step of the computation runs in the library's CUDA kernels; there is no
CPU or PyTorch fallback, and importing this package fails if the library has not
been built (``python -m min_sampling_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Union

import torch

__all__ = [
    "FsError", "lib", "LIB_PATH", "ORDER_TOP_K_FIRST", "ORDER_JOINT", "MAX_ROUNDS",
    "sampling_from_probs", "top_k_sampling", "top_p_sampling", "min_p_sampling",
    "top_k_top_p_sampling", "top_k_top_p_sampling_rng", "advance_offset",
    "top_k_top_p_sampling_pivots", "top_k_top_p_sampling_from_logits", "sampling_plan",
    "chain_speculative_sampling", "top_k_renorm_probs", "top_p_renorm_probs",
    "top_k_mask_logits", "philox4x32_10",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfs_sampling.so")
ORDER_TOP_K_FIRST = 0
ORDER_JOINT = 1
MAX_ROUNDS = 256

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_U64 = ctypes.c_uint64

_SIGNATURES = {
    "fs_sampling_from_probs": [_P, _I32, _I32, _P, _I32, _U64, _U64, _P, _P, _P, _P],
    "fs_top_k_sampling": [_P, _I32, _I32, _P, _I32, _P, _U64, _U64, _P, _P, _P, _P],
    "fs_top_p_sampling": [_P, _I32, _I32, _P, _I32, _P, _U64, _U64, _P, _P, _P, _P],
    "fs_min_p_sampling": [_P, _I32, _I32, _P, _I32, _P, _U64, _U64, _P, _P, _P, _P],
    "fs_top_k_top_p_sampling": [_P, _I32, _I32, _P, _I32, _P, _P, _P, _I32, _U64, _U64, _P, _P, _P, _P],
    "fs_top_k_top_p_sampling_rng": [_P, _I32, _I32, _P, _I32, _P, _P, _P, _I32, _P, _P, _P, _U64, _U64, _P, _P, _P,
                                    _P],
    "fs_advance_offset": [_P, _U64, _P],
    "fs_chain_speculative_sampling": [_P, _P, _P, _I32, _I32, _I32, _U64, _U64, _P, _P, _P, _P],
    "fs_sampling_plan": [_I32, _I32, _I32, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                         ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)],
    "fs_top_k_top_p_sampling_from_logits": [_P, _I32, _I32, _P, _I32, _P, _P, _P, _P, _I32, _U64, _U64, _P, _P, _P,
                                            _P],
    "fs_top_k_top_p_sampling_pivots": [_P, _I32, _I32, _P, _I32, _P, _P, _P, _I32, _I32, _U64, _U64, _P, _P, _P,
                                       _P],
    "fs_top_k_renorm_probs": [_P, _I32, _I32, _P, _P, _P, _P],
    "fs_top_p_renorm_probs": [_P, _I32, _I32, _P, _P, _P, _P],
    "fs_top_k_mask_logits": [_P, _I32, _I32, _P, _P, _P, _P],
    "fs_philox4x32_10": [_P, _P, _I64, _P, _P],
}


class FsError(RuntimeError):
    """A library call returned a status other than FS_OK."""


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m min_sampling_gb300.build` "
            "(the sampling kernels have no fallback)")
    so = ctypes.CDLL(LIB_PATH)
    for name, args in _SIGNATURES.items():
        fn = getattr(so, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    so.fs_status_string.argtypes = [_I32]
    so.fs_status_string.restype = ctypes.c_char_p
    so.fs_last_error_string.argtypes = []
    so.fs_last_error_string.restype = ctypes.c_char_p
    so.fs_max_vocab.argtypes = []
    so.fs_max_vocab.restype = _I32
    return so


_LIB: Optional[ctypes.CDLL] = None


def _lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        _LIB = _load()
    return _LIB


def __getattr__(name):
    # `lib` and `MAX_VOCAB` load the library on first access (and fail loudly if it
    # is missing), so that the build script can run inside this package.
    if name == "lib":
        return _lib()
    if name == "MAX_VOCAB":
        return int(_lib().fs_max_vocab())
    raise AttributeError(name)


def _check(status: int) -> None:
    if status != 0:
        so = _lib()
        msg = so.fs_status_string(status).decode()
        if status == 3:
            msg += " -- " + so.fs_last_error_string().decode()
        raise FsError(msg)


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _run(device, fn_name: str, *args) -> None:
    """Call a library entry with `device` made current and its current stream as the
    last argument: the library plans and launches on the current CUDA device, so the
    tensors' device must be the current one during the call."""
    with torch.cuda.device(device):
        _check(getattr(_lib(), fn_name)(*args, _stream(device)))


def _same_device(device, **tensors) -> None:
    """Every given tensor (None: absent) must live on `device`."""
    for name, t in tensors.items():
        if t is not None and t.device != device:
            raise ValueError(f"{name} is on {t.device}, but the call's tensors are on {device}")


def _ptr(t: Optional[torch.Tensor]) -> Optional[ctypes.c_void_p]:
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _matrix(x: torch.Tensor, name: str) -> torch.Tensor:
    if not isinstance(x, torch.Tensor) or x.dim() != 2:
        raise ValueError(f"{name} must be a 2-D tensor")
    if x.dtype != torch.float32 or not x.is_cuda:
        raise ValueError(f"{name} must be a float32 CUDA tensor")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return x


def _rows(v, n: int, dtype: torch.dtype, device, name: str) -> torch.Tensor:
    if isinstance(v, torch.Tensor):
        if v.shape != (n,) or v.dtype != dtype or v.device != device or not v.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [{n}] {dtype} tensor on {device}")
        return v
    return torch.full((n,), v, dtype=dtype, device=device)


def _indices(indices, b_in: int, device):
    """The output-row -> input-row map (None: one output row per input row) and the
    output batch.  The kernels read it on the device, so it must live there."""
    if indices is None:
        return None, b_in
    if not (isinstance(indices, torch.Tensor) and indices.dim() == 1 and indices.dtype == torch.int32
            and indices.device == device and indices.is_contiguous()):
        raise ValueError("indices must be a contiguous 1-D int32 tensor on the input's device")
    return indices, indices.shape[0]


def _order(order: Union[str, int]) -> int:
    if order in ("top_k_first", ORDER_TOP_K_FIRST):
        return ORDER_TOP_K_FIRST
    if order in ("joint", ORDER_JOINT):
        return ORDER_JOINT
    raise ValueError(f"order must be 'top_k_first' or 'joint', got {order!r}")


def _outputs(n: int, device):
    return (torch.empty(n, dtype=torch.int32, device=device),
            torch.empty(n, dtype=torch.uint8, device=device),
            torch.empty(n, dtype=torch.int32, device=device))


def _sample(fn_name: str, probs, indices, seed, offset, params, return_rounds, order=None):
    probs = _matrix(probs, "probs")
    b_in, V = probs.shape
    dev = probs.device
    indices, b_out = _indices(indices, b_in, dev)
    p_args = []
    for v, dtype, name in params:
        p_args.append(None if v is None else _rows(v, b_out, dtype, dev, name))
    tok, valid, rounds = _outputs(b_out, dev)
    args = [_ptr(probs), b_in, V, _ptr(indices), b_out] + [_ptr(t) for t in p_args]
    if order is not None:
        args.append(order)
    args += [int(seed) & (2 ** 64 - 1), int(offset) & (2 ** 64 - 1), _ptr(tok), _ptr(valid),
             _ptr(rounds) if return_rounds else None]
    _run(dev, fn_name, *args)
    return (tok, valid, rounds) if return_rounds else (tok, valid)


def sampling_from_probs(probs, indices=None, *, seed: int, offset: int, return_rounds: bool = False):
    """One draw per output row by inverse transform over the whole row."""
    return _sample("fs_sampling_from_probs", probs, indices, seed, offset, [], return_rounds)


def top_k_sampling(probs, top_k, indices=None, *, seed: int, offset: int, return_rounds: bool = False):
    return _sample("fs_top_k_sampling", probs, indices, seed, offset,
                   [(top_k, torch.int32, "top_k")], return_rounds)


def top_p_sampling(probs, top_p, indices=None, *, seed: int, offset: int, return_rounds: bool = False):
    return _sample("fs_top_p_sampling", probs, indices, seed, offset,
                   [(top_p, torch.float32, "top_p")], return_rounds)


def min_p_sampling(probs, min_p, indices=None, *, seed: int, offset: int, return_rounds: bool = False):
    return _sample("fs_min_p_sampling", probs, indices, seed, offset,
                   [(min_p, torch.float32, "min_p")], return_rounds)


def top_k_top_p_sampling(probs, top_k, top_p, min_p=None, order="top_k_first", indices=None, *,
                         seed: int, offset: int, return_rounds: bool = False):
    return _sample("fs_top_k_top_p_sampling", probs, indices, seed, offset,
                   [(top_k, torch.int32, "top_k"), (top_p, torch.float32, "top_p"),
                    (min_p, torch.float32, "min_p")], return_rounds, order=_order(order))


def top_k_top_p_sampling_rng(probs, top_k=None, top_p=None, min_p=None, order="joint", indices=None, *,
                             seeds=None, offsets=None, offset_dev=None, seed: int = 0, offset: int = 0,
                             return_rounds: bool = False):
    """Sampling with caller-owned generator state: per-request ``seeds`` / ``offsets``
    ([batch_out] uint64 tensors) and/or a device-resident ``offset_dev`` (one uint64,
    advanced with :func:`advance_offset`, e.g. inside a captured CUDA graph)."""
    probs = _matrix(probs, "probs")
    b_in, V = probs.shape
    dev = probs.device
    indices, b_out = _indices(indices, b_in, dev)

    def u64(t, n, name):
        if t is None:
            return None
        if not (isinstance(t, torch.Tensor) and t.dtype == torch.uint64 and t.device == dev and t.is_contiguous()
                and t.numel() == n):
            raise ValueError(f"{name} must be a contiguous uint64 tensor of {n} elements on the probs' device")
        return t

    seeds, offsets = u64(seeds, b_out, "seeds"), u64(offsets, b_out, "offsets")
    offset_dev = u64(offset_dev, 1, "offset_dev")
    ps = [None if v is None else _rows(v, b_out, dt, dev, n)
          for v, dt, n in ((top_k, torch.int32, "top_k"), (top_p, torch.float32, "top_p"),
                           (min_p, torch.float32, "min_p"))]
    tok, valid, rounds = _outputs(b_out, dev)
    _run(dev, "fs_top_k_top_p_sampling_rng",
         _ptr(probs), b_in, V, _ptr(indices), b_out, *[_ptr(t) for t in ps], _order(order), _ptr(seeds),
         _ptr(offsets), _ptr(offset_dev), int(seed) & (2 ** 64 - 1), int(offset) & (2 ** 64 - 1), _ptr(tok),
         _ptr(valid), _ptr(rounds) if return_rounds else None)
    return (tok, valid, rounds) if return_rounds else (tok, valid)


def top_k_top_p_sampling_pivots(probs, top_k=None, top_p=None, min_p=None, order="joint", indices=None, *,
                                pivots: int = 2, seed: int, offset: int, return_rounds: bool = False):
    """The sampler with the dual-pivot rule (pivots=2) or the one-pivot rule (pivots=1)."""
    probs = _matrix(probs, "probs")
    b_in, V = probs.shape
    dev = probs.device
    indices, b_out = _indices(indices, b_in, dev)
    ps = [None if v is None else _rows(v, b_out, dt, dev, n)
          for v, dt, n in ((top_k, torch.int32, "top_k"), (top_p, torch.float32, "top_p"),
                           (min_p, torch.float32, "min_p"))]
    tok, valid, rounds = _outputs(b_out, dev)
    _run(dev, "fs_top_k_top_p_sampling_pivots",
         _ptr(probs), b_in, V, _ptr(indices), b_out, *[_ptr(t) for t in ps], _order(order), int(pivots),
         int(seed) & (2 ** 64 - 1), int(offset) & (2 ** 64 - 1), _ptr(tok), _ptr(valid),
         _ptr(rounds) if return_rounds else None)
    return (tok, valid, rounds) if return_rounds else (tok, valid)


def top_k_top_p_sampling_from_logits(logits, temperature=None, top_k=None, top_p=None, min_p=None, order="joint",
                                     indices=None, *, seed: int, offset: int, return_rounds: bool = False):
    """Sampling from logits with the softmax (temperature) fused into the kernel."""
    logits = _matrix(logits, "logits")
    b_in, V = logits.shape
    dev = logits.device
    indices, b_out = _indices(indices, b_in, dev)
    ps = [None if v is None else _rows(v, b_out, dt, dev, n)
          for v, dt, n in ((temperature, torch.float32, "temperature"), (top_k, torch.int32, "top_k"),
                           (top_p, torch.float32, "top_p"), (min_p, torch.float32, "min_p"))]
    tok, valid, rounds = _outputs(b_out, dev)
    _run(dev, "fs_top_k_top_p_sampling_from_logits",
         _ptr(logits), b_in, V, _ptr(indices), b_out, *[_ptr(t) for t in ps], _order(order),
         int(seed) & (2 ** 64 - 1), int(offset) & (2 ** 64 - 1), _ptr(tok), _ptr(valid),
         _ptr(rounds) if return_rounds else None)
    return (tok, valid, rounds) if return_rounds else (tok, valid)


def chain_speculative_sampling(draft_probs, draft_tokens, target_probs, *, seed: int, offset: int):
    """Chain speculative-sampling verification: draft_probs [B, L, V] float32,
    draft_tokens [B, L] int32, target_probs [B, L + 1, V] float32 (CUDA, contiguous).
    Returns (tokens [B, L + 1] int32: the accepted drafts, the emitted token, then -1;
    accepted [B] int32; emitted [B] int32)."""
    def check3(x, name):
        if not isinstance(x, torch.Tensor) or x.dim() != 3 or x.dtype != torch.float32 or not x.is_cuda \
                or not x.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 3-D float32 CUDA tensor")
    check3(target_probs, "target_probs")
    B, L1, V = target_probs.shape
    L = L1 - 1
    if L < 0:
        raise ValueError("target_probs needs at least one row per batch entry")
    if L > 0:
        check3(draft_probs, "draft_probs")
        if tuple(draft_probs.shape) != (B, L, V):
            raise ValueError("draft_probs must be [B, L, V] with target_probs [B, L + 1, V]")
        if not isinstance(draft_tokens, torch.Tensor) or tuple(draft_tokens.shape) != (B, L):
            raise ValueError("draft_tokens must be a [B, L] tensor")
        _same_device(target_probs.device, draft_probs=draft_probs, draft_tokens=draft_tokens)
        draft_tokens = draft_tokens.to(torch.int32).contiguous()
    else:
        draft_probs = draft_tokens = None
    dev = target_probs.device
    tok = torch.empty((B, L + 1), dtype=torch.int32, device=dev)
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    emi = torch.empty(B, dtype=torch.int32, device=dev)
    _run(dev, "fs_chain_speculative_sampling",
         _ptr(draft_probs), _ptr(draft_tokens), _ptr(target_probs), B, L, V,
         int(seed) & (2 ** 64 - 1), int(offset) & (2 ** 64 - 1), _ptr(tok), _ptr(acc), _ptr(emi))
    return tok, acc, emi


def sampling_plan(batch_out: int, vocab: int, order: str = "top_k_first") -> dict:
    """CTAs per row, elements per segment, segments per CTA and CTAs per SM (at most)
    of the samplers' launch: order "top_k_first" for the top-k-first entries and
    sampling_from_probs, "joint" for the joint order and the top-k / top-p / min-p
    samplers."""
    vals = [ctypes.c_int32(0) for _ in range(4)]
    _check(_lib().fs_sampling_plan(int(batch_out), int(vocab), _order(order), *[ctypes.byref(v) for v in vals]))
    return {"cluster": vals[0].value, "segment_len": vals[1].value, "segments_per_cta": vals[2].value,
            "ctas_per_sm": vals[3].value}


def advance_offset(offset_dev, delta: int = 1) -> None:
    """*offset_dev += delta on the current stream."""
    if not (isinstance(offset_dev, torch.Tensor) and offset_dev.dtype == torch.uint64 and offset_dev.is_cuda
            and offset_dev.numel() == 1):
        raise ValueError("offset_dev must be a CUDA uint64 tensor of one element")
    _run(offset_dev.device, "fs_advance_offset", _ptr(offset_dev), int(delta) & (2 ** 64 - 1))


def _filter(fn_name, x, param, dtype, pname, out):
    x = _matrix(x, "input")
    B, V = x.shape
    p = _rows(param, B, dtype, x.device, pname)
    out = torch.empty_like(x) if out is None else _matrix(out, "out")
    if out.shape != x.shape or out.device != x.device:
        raise ValueError("out must have the input's shape and device")
    valid = torch.empty(B, dtype=torch.uint8, device=x.device)
    _run(x.device, fn_name, _ptr(x), B, V, _ptr(p), _ptr(out), _ptr(valid))
    return out, valid


def top_k_renorm_probs(probs, top_k, out=None):
    return _filter("fs_top_k_renorm_probs", probs, top_k, torch.int32, "top_k", out)


def top_p_renorm_probs(probs, top_p, out=None):
    return _filter("fs_top_p_renorm_probs", probs, top_p, torch.float32, "top_p", out)


def top_k_mask_logits(logits, top_k, out=None):
    return _filter("fs_top_k_mask_logits", logits, top_k, torch.int32, "top_k", out)


def philox4x32_10(ctr: torch.Tensor, key: torch.Tensor) -> torch.Tensor:
    """Philox4x32-10 blocks for counters [n,4] and keys [n,2] (int32/uint32 storage)."""
    if ctr.dim() != 2 or ctr.shape[1] != 4 or key.shape != (ctr.shape[0], 2):
        raise ValueError("ctr must be [n,4] and key [n,2]")
    if not (ctr.is_cuda and key.device == ctr.device and ctr.is_contiguous() and key.is_contiguous()):
        raise ValueError("ctr and key must be contiguous CUDA tensors on one device")
    if ctr.element_size() != 4 or key.element_size() != 4:
        raise ValueError("ctr and key must hold 32-bit words")
    out = torch.empty((ctr.shape[0], 4), dtype=torch.int32, device=ctr.device)
    _run(ctr.device, "fs_philox4x32_10", _ptr(ctr), _ptr(key), ctr.shape[0], _ptr(out))
    return out
