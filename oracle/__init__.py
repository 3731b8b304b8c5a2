"""Plain CPU oracle of the fused MoE layer forward (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it, and
it shares no code with the CUDA library.

The arithmetic lives in ``moe_oracle.c`` (plain loops, fp64 accumulation);
this module only compiles it with gcc and marshals numpy arrays through
ctypes.  The steps follow the compute flow of the page "用Ascend C写一个MoE
融合算子" (section "MoE的计算流程": Routing, Gating, Dispatch, Expert,
Combine); see ``moe_oracle.c`` for the citation of each step and for the
readings taken where the pages are silent.

Parity status of each function (what pins it, in ``tests/test_oracle.py``):
  router_logits  fp64 dot product vs numpy fp64 matmul; hand-derived golden.
  topk           brute-force full sort and k-pass strict argmax; exact ties.
  gate_softmax   closed forms (k=1, equal logits), sum to 1, shift invariance.
  gate_softmax_all  scipy softmax over all E (library routine as a step);
                 k = E reduces to gate_softmax; renormalised = gate_softmax.
  capacity       hand-computed values (1.2*8192*4/64 -> 615, exact integers).
  dispatch       brute-force enumerate-then-stable-sort; invariants.
  expert_ffn     identity experts (GELU(z)-GELU(-z)=z); numpy fp64 FFN with
                 math.erf; GELU fixed points.
  combine_rows   dense masked formulation; identical experts; permutation.
  combine_given  dense [T, rows] gate matrix times Y (numpy matmul as a
                 step); k = 1 with w = 1 copies rows; all dropped gives 0.
  expert_swiglu  numpy fp64 gated FFN with np.exp; SiLU fixed points; a zero
                 gate or zero up projection gives 0; swapped halves differ.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``moe_oracle.c`` into ``libmoe_oracle.so`` with gcc/OpenMP."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                                   os.path.getmtime(os.path.abspath(__file__)))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    # -ffp-contract=off: every product and sum is its own IEEE double
    # operation, as written; gcc would otherwise fuse them into FMAs on
    # aarch64 (not on x86-64), and the results would differ between machines
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.oracle_router_logits.argtypes = [I, I, I, P, P, P, P, I]
        lib.oracle_topk.argtypes = [I, I, I, P, P, P]
        lib.oracle_gate_softmax.argtypes = [I, I, P, P]
        lib.oracle_gate_softmax_all.argtypes = [I, I, I, P, P, I, P]
        lib.oracle_capacity.argtypes = [I, I, I, ctypes.c_double]
        lib.oracle_capacity.restype = ctypes.c_long
        lib.oracle_dispatch.argtypes = [I, I, I, ctypes.c_long, P, P, P, P, P]
        lib.oracle_expert_ffn.argtypes = [I, I, P, P, P, P]
        lib.oracle_combine_rows.argtypes = [I, I, I, I, I, P, P, P, P, P, P, I, P, P, I]
        lib.oracle_combine_rows_act.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, I, P, P, I]
        lib.oracle_expert_swiglu.argtypes = [I, I, P, P, P, P]
        lib.oracle_combine_given.argtypes = [I, I, I, I, P, P, P, P]
        lib.oracle_max_threads.argtypes = []
        for name in ("oracle_router_logits", "oracle_topk", "oracle_gate_softmax",
                     "oracle_gate_softmax_all",
                     "oracle_dispatch", "oracle_expert_ffn", "oracle_combine_rows",
                     "oracle_combine_rows_act", "oracle_expert_swiglu", "oracle_combine_given",
                     "oracle_max_threads"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bits(a) -> np.ndarray:
    """bf16 tensor/array -> contiguous uint16 numpy array of its bit patterns."""
    if isinstance(a, np.ndarray):
        assert a.dtype == np.uint16
        return np.ascontiguousarray(a)
    import torch  # local: torch only as a container for bf16 inputs
    assert a.dtype == torch.bfloat16
    return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def max_threads() -> int:
    return _load().oracle_max_threads()


def router_logits(x, w_router, bias=None, nthreads: int = 0) -> np.ndarray:
    """fp32 logits[T,E] = fp32(sum_h x*Wr in fp64) (+ bias in fp32)."""
    xb, wb = _bits(x), _bits(w_router)
    T, H = xb.shape
    H2, E = wb.shape
    assert H == H2
    b = None if bias is None else np.ascontiguousarray(np.asarray(bias, dtype=np.float32))
    out = np.empty((T, E), dtype=np.float32)
    _check(_load().oracle_router_logits(T, H, E, _ptr(xb), _ptr(wb), _ptr(b), _ptr(out), nthreads),
           "router_logits")
    return out


def topk(logits: np.ndarray, k: int):
    """(ids[T,k] int32, top_logits[T,k] fp32): stable descending order."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = lg.shape
    ids = np.empty((T, k), dtype=np.int32)
    vals = np.empty((T, k), dtype=np.float32)
    _check(_load().oracle_topk(T, E, k, _ptr(lg), _ptr(ids), _ptr(vals)), "topk")
    return ids, vals


def gate_softmax(top_logits: np.ndarray) -> np.ndarray:
    s = np.ascontiguousarray(top_logits, dtype=np.float32)
    T, k = s.shape
    w = np.empty((T, k), dtype=np.float32)
    _check(_load().oracle_gate_softmax(T, k, _ptr(s), _ptr(w)), "gate_softmax")
    return w


def gate_softmax_all(logits: np.ndarray, ids: np.ndarray, mode: int) -> np.ndarray:
    """Softmax over all E logits, then the k selected probabilities (mode 1)
    or those renormalised to sum 1 (mode 2)."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    idz = np.ascontiguousarray(ids, dtype=np.int32)
    T, E = lg.shape
    k = idz.shape[1]
    w = np.empty((T, k), dtype=np.float32)
    _check(_load().oracle_gate_softmax_all(T, E, k, _ptr(lg), _ptr(idz), int(mode), _ptr(w)),
           "gate_softmax_all")
    return w


def gate_weights(logits: np.ndarray, ids: np.ndarray, top_logits: np.ndarray, gating: int = 0):
    """Gate weights for gating mode 0 (softmax over the k selected), 1 or 2."""
    return gate_softmax(top_logits) if gating == 0 else gate_softmax_all(logits, ids, gating)


def capacity(T: int, k: int, E: int, capacity_factor) -> int:
    """Expert capacity, or -1 for no limit (cf None, <= 0 or NaN)."""
    cf = -1.0 if capacity_factor is None else float(capacity_factor)
    return int(_load().oracle_capacity(T, k, E, cf))


def dispatch(ids: np.ndarray, E: int, capacity_factor=None):
    """(counts[E], offsets[E+1], perm[T*k] (valid prefix offsets[E]), slot[T,k])."""
    idz = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = idz.shape
    cap = capacity(T, k, E, capacity_factor)
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.full(T * k, -1, dtype=np.int32)
    slot = np.empty((T, k), dtype=np.int32)
    _check(_load().oracle_dispatch(T, k, E, cap, _ptr(idz), _ptr(counts), _ptr(offsets),
                                   _ptr(perm), _ptr(slot)), "dispatch")
    return counts, offsets, perm, slot


def expert_ffn(xrow, w1e, w2e) -> np.ndarray:
    """GELU_erf(xrow @ W1e) @ W2e in fp64 for one row; xrow[H], W1e[H,F], W2e[F,H]."""
    xb, w1b, w2b = _bits(xrow).reshape(-1), _bits(w1e), _bits(w2e)
    H = xb.shape[0]
    F = w1b.shape[1]
    assert w1b.shape == (H, F) and w2b.shape == (F, H)
    out = np.empty(H, dtype=np.float64)
    _check(_load().oracle_expert_ffn(H, F, _ptr(xb), _ptr(w1b), _ptr(w2b), _ptr(out)), "expert_ffn")
    return out


def expert_swiglu(xrow, w1e, w2e) -> np.ndarray:
    """(SiLU(x W_gate) * (x W_up)) W_down in fp64; W1e = [gate | up] [H, 2F], W2e [F, H]."""
    xb, w1b, w2b = _bits(xrow).reshape(-1), _bits(w1e), _bits(w2e)
    H = xb.shape[0]
    F = w1b.shape[1] // 2
    assert w1b.shape == (H, 2 * F) and w2b.shape == (F, H)
    out = np.empty(H, dtype=np.float64)
    _check(_load().oracle_expert_swiglu(H, F, _ptr(xb), _ptr(w1b), _ptr(w2b), _ptr(out)),
           "expert_swiglu")
    return out


def combine_rows(x, w1, w2, ids, w, slot, rows=None, nthreads: int = 0, act: str = "gelu") -> np.ndarray:
    """y[rows] in fp64: sum over kept slots j of w[t,j] * FFN_{ids[t,j]}(x[t]).
    act "gelu": W1 [E,H,F]; "swiglu": W1 [E,H,2F] = [gate | up]; W2 [E,F,H]."""
    xb, w1b, w2b = _bits(x), _bits(w1), _bits(w2)
    T, H = xb.shape
    E, H2, F = w1b.shape
    if act == "swiglu":
        F //= 2
    assert H2 == H and w2b.shape == (E, F, H)
    idz = np.ascontiguousarray(ids, dtype=np.int32)
    k = idz.shape[1]
    wz = np.ascontiguousarray(w, dtype=np.float32)
    sz = np.ascontiguousarray(slot, dtype=np.int32)
    r = np.arange(T, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    y = np.empty((r.shape[0], H), dtype=np.float64)
    _check(_load().oracle_combine_rows_act(T, H, F, E, k, 1 if act == "swiglu" else 0, _ptr(xb),
                                           _ptr(w1b), _ptr(w2b), _ptr(idz), _ptr(wz), _ptr(sz),
                                           int(r.shape[0]), _ptr(r), _ptr(y), nthreads),
           "combine_rows")
    return y


def combine_given(Y, w: np.ndarray, slot: np.ndarray) -> np.ndarray:
    """y[t] = sum over kept j of w[t, j] * Y[slot[t, j]] in fp64; Y [n, H]
    bf16 expert outputs in dispatch order, w [T, k] fp32, slot [T, k]."""
    Yb = _bits(Y)
    n_Y, H = Yb.shape
    wz = np.ascontiguousarray(w, dtype=np.float32)
    sz = np.ascontiguousarray(slot, dtype=np.int32)
    T, k = sz.shape
    y = np.empty((T, H), dtype=np.float64)
    _check(_load().oracle_combine_given(T, H, k, n_Y, _ptr(Yb), _ptr(wz), _ptr(sz), _ptr(y)),
           "combine_given")
    return y


def route(x, w_router, k: int, bias=None, nthreads: int = 0, gating: int = 0):
    """Steps 1-2: logits, TopK ids, top logits and gate weights (all tokens)."""
    logits = router_logits(x, w_router, bias, nthreads)
    ids, vals = topk(logits, k)
    return logits, ids, vals, gate_weights(logits, ids, vals, gating)


def moe_forward(x, w_router, w1, w2, k: int, bias=None, capacity_factor=None,
                rows=None, nthreads: int = 0, gating: int = 0, act: str = "gelu") -> dict:
    """The whole layer: routing and dispatch for all tokens, FFN and combine
    for ``rows`` (all tokens when None; tokens are independent once routed)."""
    logits, ids, vals, w = route(x, w_router, k, bias, nthreads, gating)
    E = logits.shape[1]
    counts, offsets, perm, slot = dispatch(ids, E, capacity_factor)
    y = combine_rows(x, w1, w2, ids, w, slot, rows, nthreads, act)
    return dict(logits=logits, ids=ids, top_logits=vals, w=w, counts=counts,
                offsets=offsets, perm=perm, slot=slot, y=y,
                rows=np.arange(logits.shape[0]) if rows is None else np.asarray(rows))
