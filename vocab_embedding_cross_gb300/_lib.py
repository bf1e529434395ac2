"""ctypes binding of libvocabce (include/vce.h). Argument marshalling only.

Every function has the name of its C entry point and takes torch tensors (or
None for optional pointers); the tensors' device pointers and the current CUDA
stream are passed straight through. There is no fallback: if the shared
library is missing this module raises on import of the binding.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int32, c_int64, c_size_t, c_uint64, c_void_p
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libvocabce.so")

VCE_OK, VCE_ERR_ARG, VCE_ERR_UNSUPPORTED, VCE_ERR_CUDA = 0, 1, 2, 3
VCE_ERR_BAD_INDEX, VCE_ERR_TIMEOUT, VCE_ERR_WORKSPACE = 4, 5, 6
VCE_F32, VCE_BF16 = 0, 1
VCE_FLAG_ACCUMULATE_DH = 1
VCE_FLAG_DH_BF16 = 2
VCE_OP_EMBED_FWD, VCE_OP_EMBED_BWD, VCE_OP_LOSS_FWD, VCE_OP_LOSS_BWD = 0, 1, 2, 3
VCE_OP_SAMPLED_CANDIDATES = 4
VCE_OP_GREEDY_ARGMAX = 5
SIZE_MAX = (1 << 64) - 1


class VceProblem(ctypes.Structure):
    _fields_ = [("T", c_int64), ("H", c_int64), ("Vp", c_int64), ("V_real", c_int64),
                ("ignore_index", c_int64), ("S", c_int32), ("tied_weights", c_int32),
                ("dtype", c_int32), ("flags", c_int32)]


class VceError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = ""
        if status == VCE_ERR_CUDA:
            detail = " (" + lib().vce_last_error().decode() + ")"
        super().__init__(f"{where}: {status_str(status)}{detail}")


_lib = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libvocabce.so not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        P = POINTER(VceProblem)
        L.vce_workspace_size.argtypes = [P, c_int32]
        L.vce_workspace_size.restype = c_size_t
        L.vce_workspace_size_min.argtypes = [P, c_int32]
        L.vce_workspace_size_min.restype = c_size_t
        L.vce_embed_fwd.argtypes = [P, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
        L.vce_embed_fwd.restype = c_int32
        L.vce_embed_bwd.argtypes = [P, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p, c_void_p]
        L.vce_embed_bwd.restype = c_int32
        L.vce_embed_bwd_plan.argtypes = [P, c_void_p, c_void_p, c_size_t, c_void_p, c_void_p]
        L.vce_embed_bwd_plan.restype = c_int32
        L.vce_embed_bwd_apply.argtypes = [P, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p, c_void_p]
        L.vce_embed_bwd_apply.restype = c_int32
        L.vce_embed_fwd_plan.argtypes = [P, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                         c_void_p, c_void_p]
        L.vce_embed_fwd_plan.restype = c_int32
        L.vce_loss_fwd.argtypes = [P, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                   c_void_p, c_void_p, c_size_t, c_void_p, c_void_p]
        L.vce_loss_fwd.restype = c_int32
        L.vce_loss_bwd.argtypes = [P, c_void_p, c_void_p, c_void_p, c_void_p, c_float, c_void_p, c_void_p,
                                   c_void_p, c_size_t, c_void_p, c_void_p]
        L.vce_loss_bwd.restype = c_int32
        L.vce_sampled_candidates.argtypes = [P, c_void_p, c_void_p, c_int64, c_int64, c_void_p, c_void_p,
                                             c_void_p, c_void_p, c_size_t, c_void_p, c_void_p]
        L.vce_sampled_candidates.restype = c_int32
        L.vce_greedy_argmax.argtypes = [P, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                        c_void_p, c_void_p]
        L.vce_greedy_argmax.restype = c_int32
        L.vce_ngram_hash.argtypes = [c_void_p, c_int64, c_int32, c_int64, c_int64, c_int64, c_void_p, c_void_p]
        L.vce_ngram_hash.restype = c_int32
        L.vce_ngram_embed_fwd.argtypes = [P, c_void_p, c_void_p, c_void_p, c_int64, c_void_p, c_int64, c_int64,
                                          c_void_p, c_void_p, c_void_p]
        L.vce_ngram_embed_fwd.restype = c_int32
        L.vce_ngram_workspace_size.argtypes = [P]
        L.vce_ngram_workspace_size.restype = c_size_t
        L.vce_ngram_embed_bwd.argtypes = [P, c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_void_p, c_int64,
                                          c_int64, c_void_p, c_size_t, c_void_p, c_void_p]
        L.vce_ngram_embed_bwd.restype = c_int32
        L.vce_ngram_embed_bwd_plan.argtypes = [P, c_void_p, c_int64, c_int64, c_int64, c_void_p, c_size_t, c_void_p,
                                               c_void_p]
        L.vce_ngram_embed_bwd_plan.restype = c_int32
        L.vce_ngram_embed_bwd_apply.argtypes = [P, c_void_p, c_void_p, c_void_p, c_int64, c_void_p, c_int64,
                                                c_void_p, c_size_t, c_void_p, c_void_p]
        L.vce_ngram_embed_bwd_apply.restype = c_int32
        L.vce_sampled_workspace_size.argtypes = [P, c_int64]
        L.vce_sampled_workspace_size.restype = c_size_t
        L.vce_sampled_loss.argtypes = [P, c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_float,
                                       c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                       c_void_p, c_size_t, c_void_p, c_void_p]
        L.vce_sampled_loss.restype = c_int32
        L.vce_status_str.argtypes = [c_int32]
        L.vce_status_str.restype = ctypes.c_char_p
        L.vce_embed_bwd_chunk.argtypes = []
        L.vce_embed_bwd_chunk.restype = c_int32
        L.vce_version.argtypes = []
        L.vce_version.restype = c_int32
        L.vce_set_wait_limit_ns.argtypes = [c_uint64]
        L.vce_set_wait_limit_ns.restype = None
        L.vce_wait_selftest.argtypes = [c_uint64, c_void_p, c_void_p]
        L.vce_wait_selftest.restype = c_int32
        L.vce_loss_fwd_noalloc.argtypes = [P, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                           c_void_p, c_void_p, c_void_p, c_void_p]
        L.vce_loss_fwd_noalloc.restype = c_int32
        L.vce_loss_fwd_noalloc_max_scratch.argtypes = []
        L.vce_loss_fwd_noalloc_max_scratch.restype = c_size_t
        L.vce_last_error.argtypes = []
        L.vce_last_error.restype = ctypes.c_char_p
        L.vce_launch_count.argtypes = []
        L.vce_launch_count.restype = c_uint64
        L.vce_profile_begin.argtypes = [c_int32, c_void_p]
        L.vce_profile_begin.restype = c_int32
        L.vce_profile_end.argtypes = [c_void_p, c_void_p, c_int32]
        L.vce_profile_end.restype = c_int32
        _lib = L
    return _lib


def status_str(status: int) -> str:
    return lib().vce_status_str(int(status)).decode()


def problem(T: int, H: int, Vp: int, V_real: int, S: int, dtype: int, ignore_index: int = -100,
            tied: bool = False, flags: int = 0) -> VceProblem:
    return VceProblem(int(T), int(H), int(Vp), int(V_real), int(ignore_index), int(S), int(bool(tied)),
                      int(dtype), int(flags))


def _ptr(x, device=True) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if device and not x.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is not None:
        return int(stream)
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(status: int, where: str) -> None:
    if status != VCE_OK:
        raise VceError(status, where)


def vce_workspace_size(p: VceProblem, op: int) -> int:
    return int(lib().vce_workspace_size(ctypes.byref(p), op))


def vce_workspace_size_min(p: VceProblem, op: int) -> int:
    return int(lib().vce_workspace_size_min(ctypes.byref(p), op))


def vce_embed_fwd(p, ids, W, E, owner=None, local=None, dev_status=None, stream=None) -> None:
    _check(lib().vce_embed_fwd(ctypes.byref(p), _ptr(ids), _ptr(W), _ptr(E), _ptr(owner), _ptr(local),
                               _ptr(dev_status), _stream(stream)), "vce_embed_fwd")


def vce_embed_bwd(p, ids, dE, dW, ws, ws_bytes=None, dev_status=None, stream=None) -> None:
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(lib().vce_embed_bwd(ctypes.byref(p), _ptr(ids), _ptr(dE), _ptr(dW), _ptr(ws), nb,
                               _ptr(dev_status), _stream(stream)), "vce_embed_bwd")


def vce_embed_bwd_plan(p, ids, ws, ws_bytes=None, dev_status=None, stream=None) -> None:
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(lib().vce_embed_bwd_plan(ctypes.byref(p), _ptr(ids), _ptr(ws), nb, _ptr(dev_status), _stream(stream)),
           "vce_embed_bwd_plan")


def vce_embed_fwd_plan(p, ids, W, E, ws, owner=None, local=None, ws_bytes=None, dev_status=None,
                       stream=None) -> None:
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(lib().vce_embed_fwd_plan(ctypes.byref(p), _ptr(ids), _ptr(W), _ptr(E), _ptr(owner), _ptr(local),
                                    _ptr(ws), nb, _ptr(dev_status), _stream(stream)), "vce_embed_fwd_plan")


def vce_embed_bwd_apply(p, dE, dW, ws, ws_bytes=None, dev_status=None, stream=None) -> None:
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(lib().vce_embed_bwd_apply(ctypes.byref(p), _ptr(dE), _ptr(dW), _ptr(ws), nb, _ptr(dev_status),
                                     _stream(stream)), "vce_embed_bwd_apply")


def vce_loss_fwd(p, h, W, targets, loss, lse, token_loss=None, target_owner=None, max_owner=None, ws=None,
                 ws_bytes=None, dev_status=None, stream=None) -> None:
    nb = (ws.numel() * ws.element_size() if ws is not None else 0) if ws_bytes is None else ws_bytes
    _check(lib().vce_loss_fwd(ctypes.byref(p), _ptr(h), _ptr(W), _ptr(targets), _ptr(loss), _ptr(lse),
                              _ptr(token_loss), _ptr(target_owner), _ptr(max_owner), _ptr(ws), nb,
                              _ptr(dev_status), _stream(stream)), "vce_loss_fwd")


def vce_loss_bwd(p, h, W, targets, lse, g, dH, dW, ws, ws_bytes=None, dev_status=None, stream=None) -> None:
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(lib().vce_loss_bwd(ctypes.byref(p), _ptr(h), _ptr(W), _ptr(targets), _ptr(lse), float(g),
                              _ptr(dH), _ptr(dW), _ptr(ws), nb, _ptr(dev_status), _stream(stream)),
           "vce_loss_bwd")


def vce_sampled_candidates(p, targets, draws, P, cand, pos, n_unique, ws, ws_bytes=None, dev_status=None,
                           stream=None) -> None:
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    n_draws = 0 if draws is None else draws.numel()
    _check(lib().vce_sampled_candidates(ctypes.byref(p), _ptr(targets), _ptr(draws), int(n_draws), int(P),
                                        _ptr(cand), _ptr(pos), _ptr(n_unique), _ptr(ws), nb, _ptr(dev_status),
                                        _stream(stream)), "vce_sampled_candidates")


def vce_sampled_workspace_size(p: VceProblem, P: int) -> int:
    return int(lib().vce_sampled_workspace_size(ctypes.byref(p), int(P)))


def vce_sampled_loss(p, h, W, targets, draws, P, g, loss, lse, dH, dW, cand, pos, n_unique, ws, ws_bytes=None,
                     dev_status=None, stream=None) -> None:
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    n_draws = 0 if draws is None else draws.numel()
    _check(lib().vce_sampled_loss(ctypes.byref(p), _ptr(h), _ptr(W), _ptr(targets), _ptr(draws), int(n_draws),
                                  int(P), float(g), _ptr(loss), _ptr(lse), _ptr(dH), _ptr(dW), _ptr(cand),
                                  _ptr(pos), _ptr(n_unique), _ptr(ws), nb, _ptr(dev_status), _stream(stream)),
           "vce_sampled_loss")


def vce_greedy_argmax(p, h, W, argmax, max_logit=None, owner=None, ws=None, ws_bytes=None, dev_status=None,
                      stream=None) -> None:
    nb = (ws.numel() * ws.element_size() if ws is not None else 0) if ws_bytes is None else ws_bytes
    _check(lib().vce_greedy_argmax(ctypes.byref(p), _ptr(h), _ptr(W), _ptr(argmax), _ptr(max_logit), _ptr(owner),
                                   _ptr(ws), nb, _ptr(dev_status), _stream(stream)), "vce_greedy_argmax")


def vce_ngram_hash(ids, n, V, M, out, seq_len=0, stream=None) -> None:
    _check(lib().vce_ngram_hash(_ptr(ids), int(ids.numel()), int(n), int(V), int(M), int(seq_len), _ptr(out),
                                _stream(stream)), "vce_ngram_hash")


def vce_ngram_embed_fwd(p, ids, W, T2, M2, T3, M3, E, seq_len=0, dev_status=None, stream=None) -> None:
    _check(lib().vce_ngram_embed_fwd(ctypes.byref(p), _ptr(ids), _ptr(W), _ptr(T2), int(M2), _ptr(T3), int(M3),
                                     int(seq_len), _ptr(E), _ptr(dev_status), _stream(stream)),
           "vce_ngram_embed_fwd")


def vce_ngram_workspace_size(p: VceProblem) -> int:
    return int(lib().vce_ngram_workspace_size(ctypes.byref(p)))


def vce_ngram_embed_bwd(p, ids, dE, dW, dT2, M2, dT3, M3, ws, ws_bytes=None, seq_len=0, dev_status=None,
                        stream=None) -> None:
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(lib().vce_ngram_embed_bwd(ctypes.byref(p), _ptr(ids), _ptr(dE), _ptr(dW), _ptr(dT2), int(M2), _ptr(dT3),
                                     int(M3), int(seq_len), _ptr(ws), nb, _ptr(dev_status), _stream(stream)),
           "vce_ngram_embed_bwd")


def vce_ngram_embed_bwd_plan(p, ids, M2, M3, ws, ws_bytes=None, seq_len=0, dev_status=None, stream=None) -> None:
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(lib().vce_ngram_embed_bwd_plan(ctypes.byref(p), _ptr(ids), int(M2), int(M3), int(seq_len), _ptr(ws), nb,
                                          _ptr(dev_status), _stream(stream)), "vce_ngram_embed_bwd_plan")


def vce_ngram_embed_bwd_apply(p, dE, dW, dT2, M2, dT3, M3, ws, ws_bytes=None, dev_status=None,
                              stream=None) -> None:
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(lib().vce_ngram_embed_bwd_apply(ctypes.byref(p), _ptr(dE), _ptr(dW), _ptr(dT2), int(M2), _ptr(dT3),
                                           int(M3), _ptr(ws), nb, _ptr(dev_status), _stream(stream)),
           "vce_ngram_embed_bwd_apply")


def vce_embed_bwd_chunk() -> int:
    return int(lib().vce_embed_bwd_chunk())


def vce_version() -> int:
    return int(lib().vce_version())


def vce_set_wait_limit_ns(ns: int) -> None:
    lib().vce_set_wait_limit_ns(int(ns))


def vce_wait_selftest(limit_ns: int, dev_status, stream=None) -> None:
    _check(lib().vce_wait_selftest(int(limit_ns), _ptr(dev_status), _stream(stream)), "vce_wait_selftest")


KERNEL_KINDS = ["embed_gather", "embed_sort", "embed_reduce", "tc_fwd", "tc_grad", "tc_dh", "tc_dw",
                "merge", "loss_mean", "count_valid", "simt_fwd", "simt_grad", "sgemm", "wait_selftest",
                "dh_reduce", "sampled_cand", "sampled_scatter", "tc_argmax", "argmax_merge", "simt_argmax",
                "ngram_hash", "ngram_fwd", "embed_hdr", "dh_bf16", "embed_sort_cluster"]


def vce_launch_count() -> int:
    return int(lib().vce_launch_count())


def vce_profile_begin(capacity: int, stream=None) -> None:
    _check(lib().vce_profile_begin(int(capacity), _stream(stream)), "vce_profile_begin")


def vce_profile_end(capacity: int):
    """[(kernel kind name, milliseconds)] for each launch since vce_profile_begin."""
    ms = (ctypes.c_float * capacity)()
    kinds = (ctypes.c_int32 * capacity)()
    n = lib().vce_profile_end(ms, kinds, int(capacity))
    if n < 0:
        raise VceError(VCE_ERR_CUDA, "vce_profile_end")
    return [(KERNEL_KINDS[kinds[i]], float(ms[i])) for i in range(n)]


def vce_loss_fwd_noalloc(p, h, W, targets, loss, lse, token_loss=None, target_owner=None, max_owner=None,
                         dev_status=None, stream=None) -> None:
    """vce_loss_fwd with the library's fixed internal scratch instead of a workspace."""
    _check(lib().vce_loss_fwd_noalloc(ctypes.byref(p), _ptr(h), _ptr(W), _ptr(targets), _ptr(loss), _ptr(lse),
                                      _ptr(token_loss), _ptr(target_owner), _ptr(max_owner), _ptr(dev_status),
                                      _stream(stream)), "vce_loss_fwd_noalloc")


def vce_loss_fwd_noalloc_max_scratch() -> int:
    return int(lib().vce_loss_fwd_noalloc_max_scratch())
