"""GB300 speculative-sampling verify step.

Python binding of ``libspecverify.so`` (the CUDA kernels behind the C ABI in
``include/spec_verify.h``).  The functions named ``spec_verify_*`` mirror the
C entry points one to one and take raw device pointers; ``SpecVerify`` is a
convenience wrapper that takes torch tensors and only marshals arguments.
Every step of the verify computation runs in the CUDA library: there is no
Python or CPU fallback, and importing a missing library raises.
"""
from __future__ import annotations

import ctypes
import math
import os

from .build import LIBRARY

SV_OK = 0
SV_ERR_INVALID_ARG = 1
SV_ERR_SHAPE = 2
SV_ERR_DTYPE = 3
SV_ERR_CUDA = 4
SV_ERR_OOM = 5
SV_ERR_BAD_TOKEN = 6
SV_ERR_BAD_VALUE = 7
SV_ERR_TIMEOUT = 8
SV_ERR_TOO_LARGE = 9
SV_ERR_BAD_TREE = 10

SV_F32 = 0
SV_BF16 = 1

_P = ctypes.c_void_p
_I = ctypes.c_int

# (name, restype, argtypes) of every exported entry point
_SIGNATURES = [
    ("spec_verify_create", _I, [ctypes.POINTER(_P), _I, _I, _I, _I, _I]),
    ("spec_verify_run", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P]),
    ("spec_verify_run_debug", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]),
    ("spec_verify_get_status", _I, [_P]),
    ("spec_verify_set_cluster_size", _I, [_P, _I]),
    ("spec_verify_cluster_size", _I, [_P, _I, _I]),
    ("spec_verify_set_fused_logits", _I, [_P, _I]),
    ("spec_verify_error_string", ctypes.c_char_p, [_I]),
    ("spec_verify_destroy", None, [_P]),
    ("spec_verify_run_noalloc", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
    ("spec_verify_profile", _I, [_P, _I]),
    ("spec_verify_acceptance_counts", _I, [_P, ctypes.POINTER(ctypes.c_uint64), _I, _I]),
    ("spec_verify_profile_read", _I, [_P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                                      ctypes.POINTER(_I)]),
    ("spec_verify_kv_commit", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, ctypes.c_size_t, _P]),
    ("spec_verify_tree_run", _I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
    ("spec_verify_lm_head_logits", _I, [_P, _P, _I, _I, _I, _P, _P]),
    ("spec_verify_selftest_timeout", _I, [_I, ctypes.POINTER(_I), _P]),
    ("spec_verify_run_fused", _I, [_P, _P, _P, _I, _P, _P, _I, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
]

SV_KV_OVERFLOW = 1
SV_KV_BAD_COUNT = 2

_lib = None


class SpecVerifyError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: {spec_verify_error_string(status)}" if where else spec_verify_error_string(status))


def load() -> ctypes.CDLL:
    """Load the CUDA library; raises ImportError when it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIBRARY):
            raise ImportError(f"{LIBRARY} is missing: build it with "
                              "`python -m speculative_decoding_verification_49_gb300.build`")
        lib = ctypes.CDLL(LIBRARY)
        for name, res, args in _SIGNATURES:
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def exported_names():
    return [s[0] for s in _SIGNATURES]


# ---- one-to-one wrappers of the C ABI (raw pointers as Python ints) ---------

def spec_verify_create(device: int, max_B: int, max_N: int, V: int, dtype: int) -> int:
    ctx = _P()
    st = load().spec_verify_create(ctypes.byref(ctx), device, max_B, max_N, V, dtype)
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_create")
    return ctx.value


def spec_verify_run(ctx, target, draft, draft_tokens, uniforms, temperature, greedy, B, N,
                    out_tokens, num_accepted, stream) -> int:
    return load().spec_verify_run(ctx, target, draft, draft_tokens, uniforms, temperature,
                                  int(greedy), B, N, out_tokens, num_accepted, stream)


def spec_verify_run_debug(ctx, target, draft, draft_tokens, uniforms, temperature, greedy, B, N,
                          out_tokens, num_accepted, stream, q_at_draft, p_at_draft,
                          target_row_stats, draft_row_stats, ratio_at_draft=None) -> int:
    return load().spec_verify_run_debug(ctx, target, draft, draft_tokens, uniforms, temperature,
                                        int(greedy), B, N, out_tokens, num_accepted, stream,
                                        q_at_draft, p_at_draft, target_row_stats, draft_row_stats,
                                        ratio_at_draft)


def spec_verify_get_status(ctx) -> int:
    return load().spec_verify_get_status(ctx)


def spec_verify_set_cluster_size(ctx, cluster_size: int) -> int:
    return load().spec_verify_set_cluster_size(ctx, cluster_size)


def spec_verify_cluster_size(ctx, B: int, N: int) -> int:
    return load().spec_verify_cluster_size(ctx, B, N)


def spec_verify_set_fused_logits(ctx, keep: bool) -> int:
    return load().spec_verify_set_fused_logits(ctx, int(bool(keep)))


def spec_verify_error_string(status: int) -> str:
    return load().spec_verify_error_string(status).decode()


def spec_verify_destroy(ctx) -> None:
    load().spec_verify_destroy(ctx)


def spec_verify_run_noalloc(target, draft, draft_tokens, uniforms, temperature, greedy, B, N, V, dtype,
                            out_tokens, num_accepted, stream) -> int:
    """Context-free variant that allocates nothing: scratch is a fixed array
    inside the library (B <= 2048, B*(N+1) <= 16384,
    B*ceil(V*elt/4KiB) <= 32768), shared by every call on
    the device, so calls must not overlap on the GPU."""
    return load().spec_verify_run_noalloc(target, draft, draft_tokens, uniforms, temperature,
                                          int(greedy), B, N, V, dtype, out_tokens, num_accepted, stream)


def spec_verify_acceptance_counts(ctx, ncounts: int, reset: bool = False):
    """(status, counts): counts[k] sequences that accepted k drafts, the last
    entry invalid sequences."""
    arr = (ctypes.c_uint64 * ncounts)()
    st = load().spec_verify_acceptance_counts(ctx, arr, ncounts, int(bool(reset)))
    return st, list(arr)


def spec_verify_profile(ctx, enable: bool) -> int:
    return load().spec_verify_profile(ctx, int(bool(enable)))


def spec_verify_profile_read(ctx):
    """(status, ms_rows, ms_sample, runs) summed over the profiled runs."""
    a, b, n = ctypes.c_double(), ctypes.c_double(), _I()
    st = load().spec_verify_profile_read(ctx, ctypes.byref(a), ctypes.byref(b), ctypes.byref(n))
    return st, a.value, b.value, n.value


def spec_verify_tree_run(ctx, target, draft, parent, draft_tokens, uniforms, temperature, greedy, B, M,
                         out_tokens, path_nodes, num_accepted, target_row_stats, draft_row_stats, ratio_at_node,
                         stream) -> int:
    """Verify B candidate trees of M+1 nodes (device pointers; asynchronous)."""
    return load().spec_verify_tree_run(ctx, target, draft, parent, draft_tokens, uniforms, temperature,
                                       int(greedy), B, M, out_tokens, path_nodes, num_accepted,
                                       target_row_stats, draft_row_stats, ratio_at_node, stream)


def spec_verify_kv_commit(scratch, cache, cache_len, num_accepted, status, planes, B, N, max_len, row_bytes,
                          stream) -> int:
    """Append each sequence's first num_accepted scratch KV rows to its cache
    and advance cache_len (device pointers; asynchronous on stream)."""
    return load().spec_verify_kv_commit(scratch, cache, cache_len, num_accepted, status, planes, B, N,
                                        max_len, row_bytes, stream)


# ---- torch convenience wrapper -------------------------------------------------

def _ptr(t):
    return None if t is None else t.data_ptr()


class SpecVerify:
    """A context plus argument checks for torch tensors on one CUDA device.

    ``run`` enqueues the verify step on the current torch stream (or the
    given one) and returns (out_tokens [B, N+1] int32, num_accepted [B] int32)
    without synchronising.
    """

    def __init__(self, max_B: int, max_N: int, V: int, dtype: str = "bf16", device: int = 0):
        self.max_B, self.max_N, self.V, self.device = max_B, max_N, V, device
        self.dtype = dtype
        self.ctx = spec_verify_create(device, max_B, max_N, V, SV_BF16 if dtype == "bf16" else SV_F32)

    def close(self):
        if getattr(self, "ctx", None):
            spec_verify_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_cluster_size(self, c: int):
        st = spec_verify_set_cluster_size(self.ctx, c)
        if st != SV_OK:
            raise SpecVerifyError(st, "spec_verify_set_cluster_size")

    def cluster_size(self, B: int, N: int) -> int:
        return spec_verify_cluster_size(self.ctx, B, N)

    def set_fused_logits(self, keep: bool):
        """run_fused: write every verifier row's float32 logits from the
        statistics epilogue and read back the sampled rows (keep=True, the
        default), or keep them out of HBM and recompute the sampled verifier
        rows; the sampled draft rows are recomputed either way."""
        st = spec_verify_set_fused_logits(self.ctx, keep)
        if st != SV_OK:
            raise SpecVerifyError(st, "spec_verify_set_fused_logits")

    def status(self) -> int:
        return spec_verify_get_status(self.ctx)

    def acceptance_counts(self, reset: bool = False):
        """counts[k] = sequences that accepted k drafts (k = 0..max_N) since the
        last reset; counts[max_N + 1] = invalid sequences."""
        st, counts = spec_verify_acceptance_counts(self.ctx, self.max_N + 2, reset)
        if st != SV_OK:
            raise SpecVerifyError(st, "spec_verify_acceptance_counts")
        return counts

    def profile(self, enable: bool):
        st = spec_verify_profile(self.ctx, enable)
        if st != SV_OK:
            raise SpecVerifyError(st, "spec_verify_profile")

    def profile_read(self):
        """(ms in the row kernel, ms in the sampling kernel, runs)."""
        st, a, b, n = spec_verify_profile_read(self.ctx)
        if st != SV_OK:
            raise SpecVerifyError(st, "spec_verify_profile_read")
        return a, b, n

    def _check(self, target, draft, draft_tokens, uniforms, temperature, greedy):
        import torch
        want = torch.bfloat16 if self.dtype == "bf16" else torch.float32
        B, N1, V = target.shape
        N = N1 - 1
        assert V == self.V and target.dtype == want and target.is_contiguous() and target.is_cuda
        if draft is not None:
            assert draft.shape == (B, N, V) and draft.dtype == want and draft.is_contiguous()
        if draft_tokens is not None:
            assert draft_tokens.shape == (B, N) and draft_tokens.dtype == torch.int32
            assert draft_tokens.is_contiguous()
        if uniforms is not None:
            assert uniforms.shape == (B, N + 1) and uniforms.dtype == torch.float32
            assert uniforms.is_contiguous()
        if temperature is not None:
            assert temperature.shape == (B,) and temperature.dtype == torch.float32
        return B, N

    def run(self, target, draft, draft_tokens, uniforms, temperature, greedy=False,
            out_tokens=None, num_accepted=None, stream=None, debug=None):
        import torch
        B, N = self._check(target, draft, draft_tokens, uniforms, temperature, greedy)
        dev = target.device
        if out_tokens is None:
            out_tokens = torch.empty((B, N + 1), dtype=torch.int32, device=dev)
        if num_accepted is None:
            num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        args = (self.ctx, _ptr(target), _ptr(draft), _ptr(draft_tokens), _ptr(uniforms),
                _ptr(temperature), int(bool(greedy)), B, N, _ptr(out_tokens), _ptr(num_accepted),
                s.cuda_stream)
        if debug is None:
            st = spec_verify_run(*args)
        else:
            st = spec_verify_run_debug(*args, _ptr(debug.get("q_at_draft")), _ptr(debug.get("p_at_draft")),
                                       _ptr(debug.get("target_row_stats")),
                                       _ptr(debug.get("draft_row_stats")), _ptr(debug.get("ratio_at_draft")))
        if st != SV_OK:
            raise SpecVerifyError(st, "spec_verify_run")
        return out_tokens, num_accepted

    def tree_run(self, target, draft, parent, tokens, uniforms, temperature, greedy=False, out_tokens=None,
                 path_nodes=None, num_accepted=None, stream=None, stats=None):
        """Tree verification; returns (out_tokens [B, M+1], path_nodes [B, M+1],
        num_accepted [B]) without synchronising.  ``stats`` may hold
        "target_row_stats" / "draft_row_stats" float32 [B, M+1, 2] tensors and
        "ratio_at_node" float32 [B, M+1] (the ratio each tested child's
        uniform was compared with)."""
        import torch
        B, M1, V = target.shape
        M = M1 - 1
        want = torch.bfloat16 if self.dtype == "bf16" else torch.float32
        if target.dtype != want or V != self.V or not target.is_contiguous():
            raise ValueError("target logits must be contiguous [B, M+1, V] of the context's dtype")
        if draft is not None and (draft.shape != target.shape or draft.dtype != want or not draft.is_contiguous()):
            raise ValueError("draft logits must match the target's shape and dtype")
        for name, t, dt in (("parent", parent, torch.int32), ("tokens", tokens, torch.int32),
                            ("uniforms", uniforms, torch.float32)):
            if t is not None and (t.shape != (B, M + 1) or t.dtype != dt or not t.is_contiguous()):
                raise ValueError(f"{name} must be contiguous {dt} of shape ({B}, {M + 1})")
        dev = target.device
        if out_tokens is None:
            out_tokens = torch.empty((B, M + 1), dtype=torch.int32, device=dev)
        if path_nodes is None:
            path_nodes = torch.empty((B, M + 1), dtype=torch.int32, device=dev)
        if num_accepted is None:
            num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        stats = stats or {}
        st = spec_verify_tree_run(self.ctx, _ptr(target), _ptr(draft), _ptr(parent), _ptr(tokens), _ptr(uniforms),
                                  _ptr(temperature), greedy, B, M, _ptr(out_tokens), _ptr(path_nodes),
                                  _ptr(num_accepted), _ptr(stats.get("target_row_stats")),
                                  _ptr(stats.get("draft_row_stats")), _ptr(stats.get("ratio_at_node")),
                                  s.cuda_stream)
        if st != SV_OK:
            raise SpecVerifyError(st, "spec_verify_tree_run")
        return out_tokens, path_nodes, num_accepted

    def run_fused(self, target_hidden, target_weight, draft_hidden, draft_weight, draft_tokens, uniforms,
                  temperature, greedy=False, out_tokens=None, num_accepted=None, stream=None, stats=None):
        """The verify step fused into the LM-head products (context dtype
        "f32"): hidden states [rows, K] and weights [V, K] in bf16; returns
        (out_tokens, num_accepted) without synchronising."""
        import torch
        Kt = target_hidden.shape[1]
        N = draft_tokens.shape[1]
        B = target_hidden.shape[0] // (N + 1)
        Kd = draft_hidden.shape[1] if draft_hidden is not None else 0
        for t in (target_hidden, target_weight, draft_hidden, draft_weight):
            if t is not None and (t.dtype != torch.bfloat16 or not t.is_contiguous()):
                raise ValueError("hidden states and weights must be contiguous bf16")
        dev = target_hidden.device
        if out_tokens is None:
            out_tokens = torch.empty((B, N + 1), dtype=torch.int32, device=dev)
        if num_accepted is None:
            num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        stats = stats or {}
        st = load().spec_verify_run_fused(
            self.ctx, _ptr(target_hidden), _ptr(target_weight), Kt, _ptr(draft_hidden), _ptr(draft_weight), Kd,
            _ptr(draft_tokens), _ptr(uniforms), _ptr(temperature), int(bool(greedy)), B, N, _ptr(out_tokens),
            _ptr(num_accepted), _ptr(stats.get("target_row_stats")), _ptr(stats.get("draft_row_stats")),
            _ptr(stats.get("ratio_at_draft")), s.cuda_stream)
        if st != SV_OK:
            raise SpecVerifyError(st, "spec_verify_run_fused")
        return out_tokens, num_accepted

    def debug_buffers(self, B: int, N: int, device="cuda"):
        import torch
        return {
            "q_at_draft": torch.full((B, N), float("nan"), device=device),
            "p_at_draft": torch.full((B, N), float("nan"), device=device),
            "target_row_stats": torch.full((B, N + 1, 2), float("nan"), device=device),
            "draft_row_stats": torch.full((B, N, 2), float("nan"), device=device),
            "ratio_at_draft": torch.full((B, N), float("nan"), device=device),
        }


def kv_commit(scratch, cache, cache_len, num_accepted, status=None, stream=None):
    """Torch front end of spec_verify_kv_commit.

    scratch [P, B, N, *row] and cache [P, B, max_len, *row] are contiguous
    CUDA tensors of one dtype (a row is one token's entry in one plane, e.g.
    [kv_heads, head_dim]); cache_len and num_accepted are int32 [B]; status is
    an optional int32 [1] that collects SV_KV_* bits.  Enqueues on the
    current torch stream (or ``stream``) and does not synchronise."""
    import torch
    if scratch.dtype != cache.dtype or scratch.shape[:2] != cache.shape[:2] or scratch.shape[3:] != cache.shape[3:]:
        raise ValueError(f"scratch {tuple(scratch.shape)} and cache {tuple(cache.shape)} do not match")
    for name, t in (("scratch", scratch), ("cache", cache)):
        if not t.is_cuda or not t.is_contiguous() or t.dim() < 3:
            raise ValueError(f"{name} must be a contiguous CUDA tensor [P, B, rows, ...]")
    P, B, N = scratch.shape[:3]
    max_len = cache.shape[2]
    for name, t in (("cache_len", cache_len), ("num_accepted", num_accepted)):
        if t.dtype != torch.int32 or t.shape != (B,) or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor of shape ({B},)")
    row_bytes = math.prod(cache.shape[3:]) * cache.element_size()
    s = stream if stream is not None else torch.cuda.current_stream(cache.device)
    st = spec_verify_kv_commit(_ptr(scratch) if N else None, _ptr(cache), _ptr(cache_len), _ptr(num_accepted),
                               _ptr(status), P, B, N, max_len, row_bytes, s.cuda_stream)
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_kv_commit")


def lm_head_logits(hidden, weight, out=None, stream=None):
    """logits = hidden @ weight.T on the tensor cores (bf16 in, f32 out);
    hidden [M, K] and weight [V, K] contiguous bf16 CUDA tensors."""
    import torch
    if hidden.dtype != torch.bfloat16 or weight.dtype != torch.bfloat16 or hidden.dim() != 2 or weight.dim() != 2 \
            or hidden.shape[1] != weight.shape[1] or not hidden.is_contiguous() or not weight.is_contiguous():
        raise ValueError("hidden [M, K] and weight [V, K] must be contiguous bf16")
    M, K = hidden.shape
    V = weight.shape[0]
    if out is None:
        out = torch.empty((M, V), dtype=torch.float32, device=hidden.device)
    s = stream if stream is not None else torch.cuda.current_stream(hidden.device)
    st = load().spec_verify_lm_head_logits(_ptr(hidden), _ptr(weight), M, V, K, _ptr(out), s.cuda_stream)
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_lm_head_logits")
    return out


def selftest_timeout(limit_us: int = 10000, stream=None) -> bool:
    """True when a kernel wait that nothing satisfies gave up within
    limit_us and reported it (the library's bounded-wait failure detection)."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    flag = _I(0)
    st = load().spec_verify_selftest_timeout(int(limit_us), ctypes.byref(flag), s.cuda_stream)
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_selftest_timeout")
    return bool(flag.value)
