"""ctypes binding of libspecverify.so: the C ABI of include/spec_verify.h, same names.

Argument marshalling only.  Every step of the verify path runs in the CUDA
library; if the library cannot be loaded this module raises -- there is no
fallback.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

SPEC_OK = 0
SPEC_ERR_INVALID_ARG = 1
SPEC_ERR_UNSUPPORTED = 2
SPEC_ERR_MISALIGNED = 3
SPEC_ERR_WORKSPACE = 4
SPEC_ERR_CUDA = 5

SPEC_SEQ_OK = 0
SPEC_SEQ_BAD_LENGTH = 1
SPEC_SEQ_BAD_TOKEN = 2
SPEC_SEQ_BAD_UNIFORM = 3
SPEC_SEQ_NONFINITE = 4
SPEC_SEQ_EMPTY_SUPPORT = 5
SPEC_SEQ_BAD_PARAMS = 6
SPEC_SEQ_BAD_TREE = 7
SPEC_SEQ_STALLED = 8
SPEC_SEQ_ERROR_MASK = 0xFF
SPEC_SEQ_FLAG_ZERO_Q = 0x100
SPEC_SEQ_FLAG_Z_ZERO = 0x200
SPEC_SEQ_FLAG_EOS = 0x400

SPEC_BF16 = 0
SPEC_F32 = 1

# Every symbol include/spec_verify.h declares.
EXPORTED = ("spec_verify_workspace_size", "spec_verify_sample", "spec_greedy_workspace_size",
            "spec_verify_greedy", "spec_transform_probs", "spec_status_string",
            "spec_verify_sample_noalloc", "spec_verify_greedy_early", "spec_verify_sample_lenient",
            "spec_verify_workspace_size_ex", "spec_verify_sample_ex", "spec_tree_workspace_size",
            "spec_verify_greedy_tree", "spec_tree_sample_workspace_size", "spec_verify_sample_tree",
            "spec_set_early_logits_reads")


class spec_sampling_params_t(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_k", ctypes.c_int32), ("top_p", ctypes.c_float)]


class spec_verify_options_t(ctypes.Structure):
    _fields_ = [("lenience", ctypes.c_float), ("eos_token", ctypes.c_int32),
                ("target_params_seq", ctypes.c_void_p), ("draft_params_seq", ctypes.c_void_p),
                ("kept_list_only", ctypes.c_int32), ("early_exit", ctypes.c_int32)]


class SpecError(RuntimeError):
    """A non-zero spec_status_t returned by the library."""

    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} failed: {text} (status {status})")
        self.status = status


_LIB = None
vp, sz, i32, P = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, spec_sampling_params_t


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (once) and return the library, declaring every prototype."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first "
                           "(python -m speculative_decoding_verification_44_gb300.build)")
    lib = ctypes.CDLL(path)
    lib.spec_status_string.restype = ctypes.c_char_p
    lib.spec_status_string.argtypes = [ctypes.c_int]
    lib.spec_set_early_logits_reads.restype = ctypes.c_int
    lib.spec_set_early_logits_reads.argtypes = [i32]
    lib.spec_verify_workspace_size.restype = ctypes.c_int
    lib.spec_verify_workspace_size.argtypes = [i32, i32, i32, P, P, ctypes.POINTER(sz)]
    lib.spec_greedy_workspace_size.restype = ctypes.c_int
    lib.spec_greedy_workspace_size.argtypes = [i32, i32, ctypes.POINTER(sz)]
    lib.spec_verify_sample.restype = ctypes.c_int
    lib.spec_verify_sample.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp, vp, vp, P, P, i32, i32, i32,
                                       vp, sz, vp, vp, vp, vp, vp, vp]
    O = ctypes.POINTER(spec_verify_options_t)
    lib.spec_verify_workspace_size_ex.restype = ctypes.c_int
    lib.spec_verify_workspace_size_ex.argtypes = [i32, i32, i32, P, P, O, ctypes.POINTER(sz)]
    lib.spec_verify_sample_ex.restype = ctypes.c_int
    lib.spec_verify_sample_ex.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp, vp, vp, P, P, O,
                                          i32, i32, i32, vp, sz, vp, vp, vp, vp, vp, vp, vp]
    lib.spec_tree_workspace_size.restype = ctypes.c_int
    lib.spec_tree_workspace_size.argtypes = [i32, i32, ctypes.POINTER(sz)]
    lib.spec_verify_greedy_tree.restype = ctypes.c_int
    lib.spec_verify_greedy_tree.argtypes = [vp, ctypes.c_int, vp, vp, vp, i32, i32, i32, vp, sz,
                                            vp, vp, vp, vp, vp]
    lib.spec_tree_sample_workspace_size.restype = ctypes.c_int
    lib.spec_tree_sample_workspace_size.argtypes = [i32, i32, i32, P, P, ctypes.POINTER(sz)]
    lib.spec_verify_sample_tree.restype = ctypes.c_int
    lib.spec_verify_sample_tree.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp, vp, vp, P, P, i32, i32, i32, vp, sz,
                                            vp, vp, vp, vp, vp, vp, vp]
    lib.spec_verify_sample_lenient.restype = ctypes.c_int
    lib.spec_verify_sample_lenient.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp, vp, vp, P, P, ctypes.c_float,
                                               i32, i32, i32, vp, sz, vp, vp, vp, vp, vp, vp]
    lib.spec_verify_sample_noalloc.restype = ctypes.c_int
    lib.spec_verify_sample_noalloc.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp, vp, vp, P, P, i32, i32, i32,
                                               vp, vp, vp, vp, vp, vp]
    lib.spec_verify_greedy.restype = ctypes.c_int
    lib.spec_verify_greedy.argtypes = [vp, ctypes.c_int, vp, vp, i32, i32, i32, vp, sz, vp, vp, vp, vp]
    lib.spec_verify_greedy_early.restype = ctypes.c_int
    lib.spec_verify_greedy_early.argtypes = [vp, ctypes.c_int, vp, vp, i32, i32, i32, vp, sz, vp, vp, vp, vp, vp]
    lib.spec_transform_probs.restype = ctypes.c_int
    lib.spec_transform_probs.argtypes = [vp, ctypes.c_int, i32, i32, P, vp, vp, vp]
    if path == LIB_PATH:
        _LIB = lib
    return lib


def check(fn: str, status: int) -> None:
    if status != SPEC_OK:
        text = load().spec_status_string(status).decode()
        raise SpecError(fn, status, text)


def spec_status_string(status: int) -> str:
    return load().spec_status_string(status).decode()


def spec_verify_workspace_size(batch: int, gamma_max: int, vocab: int, target_params, draft_params) -> int:
    out = sz(0)
    check("spec_verify_workspace_size",
          load().spec_verify_workspace_size(batch, gamma_max, vocab, target_params, draft_params,
                                            ctypes.byref(out)))
    return out.value


def spec_verify_workspace_size_ex(batch: int, gamma_max: int, vocab: int, target_params, draft_params,
                                  options) -> int:
    out = sz(0)
    check("spec_verify_workspace_size_ex",
          load().spec_verify_workspace_size_ex(batch, gamma_max, vocab, target_params, draft_params,
                                               ctypes.byref(options) if options is not None else None,
                                               ctypes.byref(out)))
    return out.value


def spec_tree_workspace_size(batch: int, max_nodes: int) -> int:
    out = sz(0)
    check("spec_tree_workspace_size", load().spec_tree_workspace_size(batch, max_nodes, ctypes.byref(out)))
    return out.value


def spec_verify_greedy_tree(*args) -> int:
    return load().spec_verify_greedy_tree(*args)


def spec_tree_sample_workspace_size(batch: int, max_nodes: int, vocab: int, target_params, draft_params) -> int:
    out = sz(0)
    check("spec_tree_sample_workspace_size",
          load().spec_tree_sample_workspace_size(batch, max_nodes, vocab, target_params, draft_params,
                                                 ctypes.byref(out)))
    return out.value


def spec_verify_sample_tree(*args) -> int:
    return load().spec_verify_sample_tree(*args)


def spec_greedy_workspace_size(batch: int, gamma_max: int) -> int:
    out = sz(0)
    check("spec_greedy_workspace_size", load().spec_greedy_workspace_size(batch, gamma_max, ctypes.byref(out)))
    return out.value


def spec_verify_sample(*args) -> int:
    return load().spec_verify_sample(*args)


def spec_verify_sample_ex(*args) -> int:
    return load().spec_verify_sample_ex(*args)


def spec_verify_sample_lenient(*args) -> int:
    return load().spec_verify_sample_lenient(*args)


def spec_verify_sample_noalloc(*args) -> int:
    return load().spec_verify_sample_noalloc(*args)


def spec_verify_greedy(*args) -> int:
    return load().spec_verify_greedy(*args)


def spec_verify_greedy_early(*args) -> int:
    return load().spec_verify_greedy_early(*args)


def spec_transform_probs(*args) -> int:
    return load().spec_transform_probs(*args)
