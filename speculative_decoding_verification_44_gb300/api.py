"""Torch-tensor front end of the C ABI (argument marshalling only).

PyTorch here owns device memory and streams; every step of the verify path
runs in libspecverify.so.  Tensors must be CUDA tensors on the current
device, contiguous, with the layouts include/spec_verify.h documents.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib


@dataclass(frozen=True)
class SamplingParams:
    """One side's sampling rule: temperature > 0, top_k (0 = off), top_p in (0, 1] (1 = off)."""
    temperature: float = 1.0
    top_k: int = 0
    top_p: float = 1.0

    def c(self) -> _lib.spec_sampling_params_t:
        return _lib.spec_sampling_params_t(float(self.temperature), int(self.top_k), float(self.top_p))


@dataclass
class VerifyOutput:
    tokens: torch.Tensor          # [B, gamma_max+1] int32; accepted drafts, new token, then -1
    num_accepted: torch.Tensor    # [B] int32; -1 = error, commit nothing
    status: torch.Tensor          # [B] int32 SPEC_SEQ_* codes
    accept_prob: torch.Tensor | None = None   # [B, gamma_max] float32 a_i; -1 past gamma_b (early exit: past the stop)
    residual_z: torch.Tensor | None = None    # [B] float32
    num_emitted: torch.Tensor | None = None   # [B] int32 tokens committed (spec_verify_sample_ex)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return _lib.SPEC_BF16
    if t.dtype == torch.float32:
        return _lib.SPEC_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("all tensors passed to the verifier must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors passed to the verifier must be contiguous")
    return t.data_ptr()


def _stream(stream: torch.cuda.Stream | None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def set_early_logits_reads(enable: bool) -> None:
    """spec_set_early_logits_reads: let the verifiers stream their logits before they wait
    for the previous kernel in the stream (back-to-back calls overlap).  The caller guarantees
    that the kernel preceding a call has finished writing its logits when it lets its
    dependents launch (any kernel without programmatic dependent launch, or this library)."""
    _lib.check("spec_set_early_logits_reads", _lib.load().spec_set_early_logits_reads(1 if enable else 0))


def workspace_size(batch: int, gamma_max: int, vocab: int, target: SamplingParams,
                   draft: SamplingParams, per_sequence: bool = False, kept_list_only: bool = False) -> int:
    """Workspace bytes; ``per_sequence``: sized for per-sequence rules (spec_verify_workspace_size_ex),
    ``kept_list_only``: with the caller's kept-list promise."""
    if not per_sequence:
        return _lib.spec_verify_workspace_size(batch, gamma_max, vocab, target.c(), draft.c())
    opt = _lib.spec_verify_options_t(1.0, -1, 1, 1, int(kept_list_only))   # non-null per-sequence pointers
    return _lib.spec_verify_workspace_size_ex(batch, gamma_max, vocab, target.c(), draft.c(), opt)


def rules_tensor(rules, device) -> torch.Tensor:
    """Per-sequence sampling rules as the [B] spec_sampling_params_t array the C ABI reads
    (int32 [B, 3]: temperature bits, top_k, top_p bits) on ``device``."""
    t = torch.tensor([[r.temperature, 0.0, r.top_p] for r in rules], dtype=torch.float32).view(torch.int32)
    t[:, 1] = torch.tensor([int(r.top_k) for r in rules], dtype=torch.int32)
    return t.contiguous().to(device)


def greedy_workspace_size(batch: int, gamma_max: int) -> int:
    return _lib.spec_greedy_workspace_size(batch, gamma_max)


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled workspace (the library needs zeros before first use and restores them)."""
    return torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)


def alloc_outputs(batch: int, gamma_max: int, device, accept_prob: bool = True,
                  residual_z: bool = True) -> VerifyOutput:
    return VerifyOutput(
        tokens=torch.empty(batch, gamma_max + 1, dtype=torch.int32, device=device),
        num_accepted=torch.empty(batch, dtype=torch.int32, device=device),
        status=torch.empty(batch, dtype=torch.int32, device=device),
        accept_prob=torch.empty(batch, gamma_max, dtype=torch.float32, device=device) if accept_prob else None,
        residual_z=torch.empty(batch, dtype=torch.float32, device=device) if residual_z else None)


def verify_sample(target_logits: torch.Tensor, draft_logits: torch.Tensor | None,
                  draft_tokens: torch.Tensor, u_accept: torch.Tensor, u_sample: torch.Tensor,
                  target: SamplingParams, draft: SamplingParams,
                  gamma_per_seq: torch.Tensor | None = None,
                  draft_is_onehot: torch.Tensor | None = None,
                  workspace: torch.Tensor | None = None, out: VerifyOutput | None = None,
                  stream: torch.cuda.Stream | None = None,
                  lenience: float | None = None, eos_token: int | None = None,
                  target_rules=None, draft_rules=None, kept_list_only: bool = False,
                  early_exit: bool = False) -> VerifyOutput:
    """spec_verify_sample on torch tensors; spec_verify_sample_lenient when only
    ``lenience`` is given; spec_verify_sample_ex when ``eos_token``, per-sequence
    rules or ``early_exit`` are given.

    target_logits [B, G+1, V] and draft_logits [B, G, V] (or None: all one-hot) of
    bfloat16 / float32; draft_tokens [B, G] int32; u_accept [B, G] and u_sample [B]
    float32; gamma_per_seq [B] int32; draft_is_onehot [B] uint8; lenience in (0, 1];
    target_rules / draft_rules: per-sequence rules, a list of SamplingParams or a
    tensor from rules_tensor() (the scalar ``target`` / ``draft`` then only size the call);
    kept_list_only: the promise that every per-sequence rule has 1 <= top_k <= 128;
    early_exit: positions in order, each sequence stopping at its first failed row
    or rejected draft (rows after it may be skipped).
    """
    B, G1, V = target_logits.shape
    G = G1 - 1
    if draft_logits is not None and draft_logits.dtype != target_logits.dtype:
        raise TypeError("target and draft logits must share a dtype")
    dev = target_logits.device
    ex = eos_token is not None or target_rules is not None or draft_rules is not None or early_exit
    if isinstance(target_rules, (list, tuple)):
        target_rules = rules_tensor(target_rules, dev)
    if isinstance(draft_rules, (list, tuple)):
        draft_rules = rules_tensor(draft_rules, dev)
    if workspace is None:
        workspace = new_workspace(workspace_size(B, G, V, target, draft,
                                                 per_sequence=target_rules is not None or draft_rules is not None,
                                                 kept_list_only=kept_list_only), dev)
    if out is None:
        out = alloc_outputs(B, G, dev)
    if ex and out.num_emitted is None:
        out.num_emitted = torch.empty(B, dtype=torch.int32, device=dev)
    head = (_ptr(target_logits), _ptr(draft_logits), _dtype_code(target_logits), _ptr(draft_tokens),
            _ptr(gamma_per_seq), _ptr(draft_is_onehot), _ptr(u_accept), _ptr(u_sample),
            target.c(), draft.c())
    tail = (B, G, V, _ptr(workspace), workspace.numel(),
            _ptr(out.tokens), _ptr(out.num_accepted), _ptr(out.accept_prob), _ptr(out.residual_z),
            _ptr(out.status), _stream(stream))
    if ex:
        opt = _lib.spec_verify_options_t(1.0 if lenience is None else float(lenience),
                                         -1 if eos_token is None else int(eos_token),
                                         _ptr(target_rules), _ptr(draft_rules), int(kept_list_only),
                                         int(bool(early_exit)))
        _lib.check("spec_verify_sample_ex",
                   _lib.spec_verify_sample_ex(*head, ctypes.byref(opt), *tail[:-1], _ptr(out.num_emitted), tail[-1]))
    elif lenience is None:
        _lib.check("spec_verify_sample", _lib.spec_verify_sample(*head, *tail))
    else:
        _lib.check("spec_verify_sample_lenient",
                   _lib.spec_verify_sample_lenient(*head, float(lenience), *tail))
    return out


def verify_greedy(target_logits: torch.Tensor, draft_tokens: torch.Tensor,
                  gamma_per_seq: torch.Tensor | None = None,
                  workspace: torch.Tensor | None = None, out: VerifyOutput | None = None,
                  stream: torch.cuda.Stream | None = None) -> VerifyOutput:
    """spec_verify_greedy on torch tensors (target_logits [B, G+1, V])."""
    B, G1, V = target_logits.shape
    G = G1 - 1
    dev = target_logits.device
    if workspace is None:
        workspace = new_workspace(greedy_workspace_size(B, G), dev)
    if out is None:
        out = alloc_outputs(B, G, dev, accept_prob=False, residual_z=False)
    st = _lib.spec_verify_greedy(
        _ptr(target_logits), _dtype_code(target_logits), _ptr(draft_tokens), _ptr(gamma_per_seq),
        B, G, V, _ptr(workspace), workspace.numel(), _ptr(out.tokens), _ptr(out.num_accepted),
        _ptr(out.status), _stream(stream))
    _lib.check("spec_verify_greedy", st)
    return out


def verify_greedy_early(target_logits: torch.Tensor, draft_tokens: torch.Tensor,
                        gamma_per_seq: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None, out: VerifyOutput | None = None,
                        rows_read: torch.Tensor | None = None,
                        stream: torch.cuda.Stream | None = None) -> VerifyOutput:
    """spec_verify_greedy_early on torch tensors: rows after the first mismatch are
    skipped.  ``rows_read`` ([B] int32), if given, receives the rows read."""
    B, G1, V = target_logits.shape
    G = G1 - 1
    dev = target_logits.device
    if workspace is None:
        workspace = new_workspace(greedy_workspace_size(B, G), dev)
    if out is None:
        out = alloc_outputs(B, G, dev, accept_prob=False, residual_z=False)
    st = _lib.spec_verify_greedy_early(
        _ptr(target_logits), _dtype_code(target_logits), _ptr(draft_tokens), _ptr(gamma_per_seq),
        B, G, V, _ptr(workspace), workspace.numel(), _ptr(out.tokens), _ptr(out.num_accepted),
        _ptr(out.status), _ptr(rows_read), _stream(stream))
    _lib.check("spec_verify_greedy_early", st)
    return out


def tree_workspace_size(batch: int, max_nodes: int) -> int:
    return _lib.spec_tree_workspace_size(batch, max_nodes)


def verify_greedy_tree(target_logits: torch.Tensor, tree_tokens: torch.Tensor, tree_parents: torch.Tensor,
                       nodes_per_seq: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                       out: VerifyOutput | None = None, path: torch.Tensor | None = None,
                       stream: torch.cuda.Stream | None = None) -> tuple[VerifyOutput, torch.Tensor]:
    """spec_verify_greedy_tree on torch tensors: target_logits [B, N, V], tree_tokens and
    tree_parents [B, N] int32, nodes_per_seq [B] int32.  Returns the outputs (tokens [B, N])
    and the accepted path's nodes [B, N]."""
    B, N, V = target_logits.shape
    dev = target_logits.device
    if workspace is None:
        workspace = new_workspace(tree_workspace_size(B, N), dev)
    if out is None:
        out = VerifyOutput(tokens=torch.empty(B, N, dtype=torch.int32, device=dev),
                           num_accepted=torch.empty(B, dtype=torch.int32, device=dev),
                           status=torch.empty(B, dtype=torch.int32, device=dev))
    if path is None:
        path = torch.empty(B, N, dtype=torch.int32, device=dev)
    st = _lib.spec_verify_greedy_tree(
        _ptr(target_logits), _dtype_code(target_logits), _ptr(tree_tokens), _ptr(tree_parents),
        _ptr(nodes_per_seq), B, N, V, _ptr(workspace), workspace.numel(), _ptr(out.tokens),
        _ptr(out.num_accepted), _ptr(path), _ptr(out.status), _stream(stream))
    _lib.check("spec_verify_greedy_tree", st)
    return out, path


def tree_sample_workspace_size(batch: int, max_nodes: int, vocab: int, target: SamplingParams,
                                draft: SamplingParams) -> int:
    return _lib.spec_tree_sample_workspace_size(batch, max_nodes, vocab, target.c(), draft.c())


def verify_sample_tree(target_logits: torch.Tensor, draft_logits: torch.Tensor, tree_tokens: torch.Tensor,
                       tree_parents: torch.Tensor, u_node: torch.Tensor, u_sample: torch.Tensor,
                       target_params: SamplingParams, draft_params: SamplingParams,
                       nodes_per_seq: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                       out: VerifyOutput | None = None, path: torch.Tensor | None = None,
                       stream: torch.cuda.Stream | None = None) -> tuple[VerifyOutput, torch.Tensor]:
    """spec_verify_sample_tree on torch tensors: target_logits and draft_logits [B, N, V],
    tree_tokens and tree_parents [B, N] int32, u_node [B, N] and u_sample [B] float32,
    nodes_per_seq [B] int32.  Returns the outputs (tokens [B, N], accept_prob [B, N - 1])
    and the accepted path's nodes [B, N]."""
    B, N, V = target_logits.shape
    dev = target_logits.device
    if workspace is None:
        workspace = new_workspace(tree_sample_workspace_size(B, N, V, target_params, draft_params), dev)
    if out is None:
        out = VerifyOutput(tokens=torch.empty(B, N, dtype=torch.int32, device=dev),
                           num_accepted=torch.empty(B, dtype=torch.int32, device=dev),
                           status=torch.empty(B, dtype=torch.int32, device=dev),
                           accept_prob=torch.empty(B, max(N - 1, 1), dtype=torch.float32, device=dev),
                           residual_z=torch.empty(B, dtype=torch.float32, device=dev))
    if path is None:
        path = torch.empty(B, N, dtype=torch.int32, device=dev)
    st = _lib.spec_verify_sample_tree(
        _ptr(target_logits), _ptr(draft_logits), _dtype_code(target_logits), _ptr(tree_tokens),
        _ptr(tree_parents), _ptr(nodes_per_seq), _ptr(u_node), _ptr(u_sample), target_params.c(),
        draft_params.c(), B, N, V, _ptr(workspace), workspace.numel(), _ptr(out.tokens), _ptr(out.num_accepted),
        _ptr(path), _ptr(out.accept_prob), _ptr(out.residual_z), _ptr(out.status), _stream(stream))
    _lib.check("spec_verify_sample_tree", st)
    return out, path


def transform_probs(logits: torch.Tensor, params: SamplingParams,
                    stream: torch.cuda.Stream | None = None) -> tuple[torch.Tensor, torch.Tensor]:
    """spec_transform_probs: full probability rows of a [rows, V] logits tensor."""
    rows, V = logits.reshape(-1, logits.shape[-1]).shape
    flat = logits.reshape(rows, V)
    probs = torch.empty(rows, V, dtype=torch.float32, device=logits.device)
    status = torch.empty(rows, dtype=torch.int32, device=logits.device)
    st = _lib.spec_transform_probs(_ptr(flat), _dtype_code(flat), rows, V, params.c(), _ptr(probs),
                                   _ptr(status), _stream(stream))
    _lib.check("spec_transform_probs", st)
    return probs.reshape(*logits.shape[:-1], V), status.reshape(logits.shape[:-1])


class BoundSample:
    """A spec_verify_sample call with its buffers marshalled once.

    For serving loops that reuse the same device buffers every step: the
    arguments are validated and converted at construction, and each call is one
    C-ABI call on the stream current at construction (or the one given).
    Writes into ``self.out``; raises on a non-zero status.
    """

    def __init__(self, target_logits, draft_logits, draft_tokens, u_accept, u_sample,
                 target: SamplingParams, draft: SamplingParams, gamma_per_seq=None,
                 draft_is_onehot=None, workspace=None, out=None, stream=None, lenience=None,
                 eos_token=None, target_rules=None, draft_rules=None, kept_list_only=False,
                 early_exit=False):
        B, G1, V = target_logits.shape
        G = G1 - 1
        dev = target_logits.device
        if draft_logits is not None and draft_logits.dtype != target_logits.dtype:
            raise TypeError("target and draft logits must share a dtype")
        if isinstance(target_rules, (list, tuple)):
            target_rules = rules_tensor(target_rules, dev)
        if isinstance(draft_rules, (list, tuple)):
            draft_rules = rules_tensor(draft_rules, dev)
        per = target_rules is not None or draft_rules is not None
        ex = per or eos_token is not None or bool(early_exit)
        self.workspace = workspace if workspace is not None else new_workspace(
            workspace_size(B, G, V, target, draft, per_sequence=per, kept_list_only=kept_list_only), dev)
        self.out = out if out is not None else alloc_outputs(B, G, dev)
        if ex and self.out.num_emitted is None:
            self.out.num_emitted = torch.empty(B, dtype=torch.int32, device=dev)
        self._keep = (target_logits, draft_logits, draft_tokens, u_accept, u_sample, gamma_per_seq,
                      draft_is_onehot, target_rules, draft_rules)
        o = self.out
        head = (_ptr(target_logits), _ptr(draft_logits), _dtype_code(target_logits),
                _ptr(draft_tokens), _ptr(gamma_per_seq), _ptr(draft_is_onehot), _ptr(u_accept),
                _ptr(u_sample), target.c(), draft.c())
        tail = (B, G, V, _ptr(self.workspace), self.workspace.numel(), _ptr(o.tokens), _ptr(o.num_accepted),
                _ptr(o.accept_prob), _ptr(o.residual_z), _ptr(o.status))
        lib = _lib.load()
        if ex:
            self._opt = _lib.spec_verify_options_t(1.0 if lenience is None else float(lenience),
                                                   -1 if eos_token is None else int(eos_token),
                                                   _ptr(target_rules), _ptr(draft_rules), int(kept_list_only),
                                                   int(bool(early_exit)))
            self._fn, self._name = lib.spec_verify_sample_ex, "spec_verify_sample_ex"
            self._args = (*head, ctypes.byref(self._opt), *tail, _ptr(o.num_emitted), _stream(stream))
        elif lenience is not None:
            self._fn, self._name = lib.spec_verify_sample_lenient, "spec_verify_sample_lenient"
            self._args = (*head, float(lenience), *tail, _stream(stream))
        else:
            self._fn, self._name = lib.spec_verify_sample, "spec_verify_sample"
            self._args = (*head, *tail, _stream(stream))

    def __call__(self) -> VerifyOutput:
        st = self._fn(*self._args)
        if st:
            _lib.check(self._name, st)
        return self.out
