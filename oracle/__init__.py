"""Float64 CPU oracle of the speculative-sampling verify step.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` are the only callers.  The
product (the CUDA library and its binding) never imports this package.

The arithmetic lives in ``sv_oracle.c`` (plain C, double precision); this
module compiles it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "sv_oracle.c")
LIBRARY = os.path.join(HERE, "liboracle.so")

DTYPES = {"f32": 0, "bf16": 1, "f64": 2}
SEQ_BAD_TOKEN = 1
SEQ_BAD_VALUE = 2

_lock = threading.Lock()


def compile_library(source: str = SOURCE, out: str = LIBRARY) -> str:
    """Compile the oracle with gcc.  FMA contraction is off so that x86 and
    aarch64 hosts round identically."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, source, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build() -> str:
    return compile_library()


def _stale(lib: str, src: str) -> bool:
    return (not os.path.exists(lib)) or os.path.getmtime(lib) < os.path.getmtime(src)


def _as_logits(x, dtype: str) -> np.ndarray:
    """Raw logits as a C-contiguous numpy array of the oracle's storage type.
    bf16 is passed as its uint16 bit pattern."""
    if hasattr(x, "detach"):  # torch tensor
        import torch
        t = x.detach().to("cpu").contiguous()
        if dtype == "bf16":
            assert t.dtype == torch.bfloat16
            return t.view(torch.int16).numpy().view(np.uint16)
        x = t.numpy()
    x = np.ascontiguousarray(x)
    want = {"f32": np.float32, "bf16": np.uint16, "f64": np.float64}[dtype]
    assert x.dtype == want, (x.dtype, dtype)
    return x


def _np(x, dt):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=dt))


class Oracle:
    """ctypes handle on one compiled oracle library."""

    def __init__(self, lib_path: str | None = None):
        if lib_path is None:
            with _lock:
                if _stale(LIBRARY, SOURCE):
                    compile_library()
            lib_path = LIBRARY
        self.lib = ctypes.CDLL(lib_path)
        P = ctypes.c_void_p
        i = ctypes.c_int
        self.lib.orc_verify.restype = i
        self.lib.orc_verify.argtypes = [P, P, i, P, P, P, i, i, i, i, P, P,
                                        P, P, P, P, P, P, P, P, i]
        self.lib.orc_softmax_row.restype = i
        self.lib.orc_softmax_row.argtypes = [P, i, i, ctypes.c_double, P, P, P]
        self.lib.orc_tree_verify.restype = i
        self.lib.orc_tree_verify.argtypes = [P, P, i, P, P, P, P, i, i, i, i, P, P, P, P, P, P, P, P, P, i]
        self.lib.orc_kv_commit.restype = i
        self.lib.orc_kv_commit.argtypes = [P, P, P, P, i, i, i, i, ctypes.c_size_t]

    def verify(self, target, draft, draft_tokens, uniforms, temperature=None,
               greedy=False, dtype="f32", threads=1, diagnostics=True):
        """Run the verify step on B sequences.

        target: [B, N+1, V] logits, draft: [B, N, V] logits (may be None when
        greedy), draft_tokens: [B, N] int, uniforms: [B, N+1] (float32 values
        are widened exactly), temperature: [B] or None when greedy.

        Returns a dict of numpy arrays: out_tokens [B, N+1], num_accepted [B],
        seq_status [B] and, with diagnostics, q_at_d / p_at_d [B, N],
        tstats [B, N+1, 2], dstats [B, N, 2], accept_margin [B, N],
        sample_margin [B] and ratio_at_d [B, N] (q(d)/p(d) of every accept
        test made, +inf where p(d) == 0, NaN where no test was made).
        """
        tgt = _as_logits(target, dtype)
        B, N1, V = tgt.shape
        N = N1 - 1
        drf = None if draft is None else _as_logits(draft, dtype)
        if drf is not None:
            assert drf.shape == (B, N, V), drf.shape
        tok = _np(draft_tokens, np.int32)
        if tok is None:
            tok = np.zeros((B, N), np.int32)
        assert tok.shape == (B, N)
        u = _np(uniforms, np.float64)
        assert u.shape == (B, N + 1)
        T = _np(temperature, np.float64)
        if T is not None:
            assert T.shape == (B,)
        out = np.full((B, N + 1), -7, np.int32)
        acc = np.full((B,), -7, np.int32)
        st = np.zeros((B,), np.int32)
        res = {"out_tokens": out, "num_accepted": acc, "seq_status": st}
        if diagnostics:
            res.update(
                q_at_d=np.full((B, N), np.nan), p_at_d=np.full((B, N), np.nan),
                tstats=np.full((B, N + 1, 2), np.nan), dstats=np.full((B, N, 2), np.nan),
                accept_margin=np.full((B, N), np.nan), sample_margin=np.full((B,), np.nan),
                ratio_at_d=np.full((B, N), np.nan))

        def ptr(a):
            return None if a is None else a.ctypes.data

        rc = self.lib.orc_verify(
            ptr(tgt), ptr(drf), DTYPES[dtype], ptr(tok), ptr(u), ptr(T),
            int(bool(greedy)), B, N, V, ptr(out), ptr(acc),
            ptr(res.get("q_at_d")), ptr(res.get("p_at_d")),
            ptr(res.get("tstats")), ptr(res.get("dstats")),
            ptr(res.get("accept_margin")), ptr(res.get("sample_margin")),
            ptr(st), ptr(res.get("ratio_at_d")), int(threads))
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        return res

    def softmax_row(self, row, T, dtype="f64"):
        """softmax(row / T) with its normaliser (m, S)."""
        z = _as_logits(row, dtype)
        V = z.shape[0]
        probs = np.empty(V, np.float64)
        m = ctypes.c_double()
        S = ctypes.c_double()
        rc = self.lib.orc_softmax_row(z.ctypes.data, DTYPES[dtype], V, float(T),
                                      probs.ctypes.data, ctypes.byref(m), ctypes.byref(S))
        if rc != 0:
            raise ValueError("bad softmax arguments")
        return probs, m.value, S.value


    def tree_verify(self, target, draft, parent, tokens, uniforms, temperature=None,
                    greedy=False, dtype="f32", threads=1, diagnostics=True):
        """Verify B candidate trees of M+1 nodes (node 0 = the committed context).

        target, draft: [B, M+1, V] logits per node (draft rows of leaves are
        not read; draft may be None when greedy); parent: [B, M+1] or [M+1]
        int (parent[0] = -1, parent[n] < n); tokens: [B, M+1] int (entry 0
        unused); uniforms: [B, M+1] (entry n >= 1 the accept test of node n,
        entry 0 the final sample); temperature: [B] or None when greedy.

        Returns out_tokens, path_nodes [B, M+1], num_accepted, seq_status [B]
        and, with diagnostics, tstats / dstats [B, M+1, 2] (visited nodes),
        accept_margin [B, M+1] (NaN = not tested), sample_margin [B] and
        ratio_at [B, M+1] (r(x)/p(x) of each tested child, +inf where
        p(x) == 0, NaN = not tested)."""
        tgt = _as_logits(target, dtype)
        B, M1, V = tgt.shape
        M = M1 - 1
        drf = None if draft is None else _as_logits(draft, dtype)
        if drf is not None:
            assert drf.shape == (B, M + 1, V), drf.shape
        par = _np(parent, np.int32)
        if par.ndim == 1:
            par = np.ascontiguousarray(np.broadcast_to(par, (B, M + 1)))
        tok = _np(tokens, np.int32)
        u = _np(uniforms, np.float64)
        T = _np(temperature, np.float64)
        assert par.shape == (B, M + 1) and tok.shape == (B, M + 1) and u.shape == (B, M + 1)
        res = {"out_tokens": np.full((B, M + 1), -7, np.int32), "path_nodes": np.full((B, M + 1), -7, np.int32),
               "num_accepted": np.full((B,), -7, np.int32), "seq_status": np.zeros((B,), np.int32)}
        if diagnostics:
            res.update(tstats=np.full((B, M + 1, 2), np.nan), dstats=np.full((B, M + 1, 2), np.nan),
                       accept_margin=np.full((B, M + 1), np.nan), sample_margin=np.full((B,), np.nan),
                       ratio_at=np.full((B, M + 1), np.nan))

        def ptr(a):
            return None if a is None else a.ctypes.data

        rc = self.lib.orc_tree_verify(
            ptr(tgt), ptr(drf), DTYPES[dtype], ptr(par), ptr(tok), ptr(u), ptr(T), int(bool(greedy)),
            B, M, V, ptr(res["out_tokens"]), ptr(res["path_nodes"]), ptr(res["num_accepted"]),
            ptr(res.get("tstats")), ptr(res.get("dstats")), ptr(res.get("accept_margin")),
            ptr(res.get("sample_margin")), ptr(res["seq_status"]), ptr(res.get("ratio_at")), int(threads))
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        return res

    def kv_commit(self, scratch, cache, cache_len, num_accepted):
        """Append each sequence's accepted draft KV rows to its cache.

        scratch: uint8 [P, B, N, row_bytes], cache: uint8 [P, B, max_len,
        row_bytes], cache_len: int [B], num_accepted: int [B].  Works on
        copies; returns (cache, cache_len, status bits)."""
        s = np.ascontiguousarray(_np(scratch, np.uint8))
        c = np.array(_np(cache, np.uint8), copy=True, order="C")
        ln = np.array(_np(cache_len, np.int32), copy=True)
        a = _np(num_accepted, np.int32)
        P, B, N, row = s.shape
        assert c.shape[:2] == (P, B) and c.shape[3] == row, (c.shape, s.shape)
        assert ln.shape == (B,) and a.shape == (B,)
        st = self.lib.orc_kv_commit(s.ctypes.data, c.ctypes.data, ln.ctypes.data, a.ctypes.data,
                                    P, B, N, c.shape[2], row)
        return c, ln, int(st)


_default: Oracle | None = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def verify(*args, **kwargs):
    return default().verify(*args, **kwargs)


def kv_commit(*args, **kwargs):
    return default().kv_commit(*args, **kwargs)


def tree_verify(*args, **kwargs):
    return default().tree_verify(*args, **kwargs)


def lm_head_logits(hidden, weight):
    """logits[r, v] = sum_k hidden[r, k] * weight[v, k] in float64 (the plain
    definition of the LM-head product; bf16 inputs widen exactly)."""
    h = np.asarray(hidden.float().cpu().numpy() if hasattr(hidden, "float") else hidden, dtype=np.float64)
    w = np.asarray(weight.float().cpu().numpy() if hasattr(weight, "float") else weight, dtype=np.float64)
    return h @ w.T
