"""Seeded synthetic workloads for the Vegas hot path (test and benchmark input).

This package only *draws inputs*: queries, keys, values, heavy-hitter position
sets and ragged lengths, as bf16 bit patterns (numpy ``uint16``).  It holds no
attention, scoring or selection arithmetic, so both the CPU oracle's callers and
the CUDA path's callers can take their inputs from here.

The five workloads restate the shapes of the evaluation settings described on the
Vegas page (Qwen3 / gpt-oss-class models, contexts up to 128K tokens; Vegas §4)
with synthetic data, since no weights or datasets are available:

* ``tiny``      B=1, H_q=8, H_kv=2, d=64, n=512, gamma=3, k=64, i.i.d. N(0,1).
* ``llama8b``   B=1, H_q=32, H_kv=8, d=128, n=32768, gamma=7, k=2048, 2 % heavy hitters.
* ``batched``   B=16, n=16384, gamma=7, k=1024, heavy hitters with one u per sequence,
                selection on all gamma+1 rows and Collect-2-Query beside it.
* ``long70b``   B=1, H_q=64, H_kv=8, d=128, n=131072, gamma=5, k=4096, 1 % heavy hitters
                and 16 attention sinks.
* ``loop32``    32 layers of llama8b heads, B=8, ragged n ~ U[4096, 65536], gamma=6, k=2048.

Every value is a pure function of (seed, stream, index) (see ``gen.c``), so a slice
of a tensor can be regenerated alone: the tests regenerate just the sequences and
heads they sample at full size.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libvgsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gen.c`` into ``_build/libvgsynth.so`` (gcc, OpenMP, no FMA contraction)."""
    src = os.path.join(_HERE, "gen.c")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src)):
        return _LIB_PATH
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i64, i32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int
            vp = ctypes.c_void_p
            lib.vgs_fill_normal.argtypes = [u64, u64, u64, i64, vp]
            lib.vgs_unit_vector.argtypes = [u64, u64, i32, vp]
            lib.vgs_fill_keys.argtypes = [u64, u64, i64, i64, i32, i32, vp, vp, vp]
            lib.vgs_fill_query.argtypes = [u64, u64, u64, i64, i32, vp, vp]
            lib.vgs_choose.argtypes = [u64, u64, i64, i64, i64, ctypes.c_uint8, vp]
            lib.vgs_choose.restype = i32
            lib.vgs_uniform_int.argtypes = [u64, u64, u64, i64, i64]
            lib.vgs_uniform_int.restype = i64
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- stream ids
T_K, T_V, T_QV, T_KNEW, T_VNEW, T_QD, T_KD, T_VD, T_U, T_HEAVY, T_LEN = range(1, 12)


def stream_id(tensor: int, layer: int = 0, b: int = 0) -> int:
    """Independent stream per (tensor, layer, sequence)."""
    return (tensor << 48) | (layer << 24) | b


# ---------------------------------------------------------------- primitives
def normal_bf16(seed: int, stream: int, count: int, start: int = 0) -> np.ndarray:
    out = np.empty(count, dtype=np.uint16)
    _load().vgs_fill_normal(seed, stream, start, count, _ptr(out))
    return out


def unit_vector(seed: int, stream: int, d: int) -> np.ndarray:
    out = np.empty(d, dtype=np.float32)
    _load().vgs_unit_vector(seed, stream, d, _ptr(out))
    return out


def keys_bf16(seed, stream, start_pos, npos, H, d, kind=None, u=None) -> np.ndarray:
    out = np.empty((npos, H, d), dtype=np.uint16)
    if kind is not None:
        kind = np.ascontiguousarray(kind, dtype=np.uint8)
        assert kind.shape == (npos,)
        if u is None and kind.any():
            raise ValueError("heavy-hitter or sink keys need the direction u")
    if u is not None:
        u = np.ascontiguousarray(u, dtype=np.float32)
    _load().vgs_fill_keys(seed, stream, start_pos, npos, H, d, _ptr(kind), _ptr(u), _ptr(out))
    return out


def query_bf16(seed, stream, count, d, u=None, start=0) -> np.ndarray:
    out = np.empty(count, dtype=np.uint16)
    if u is not None:
        u = np.ascontiguousarray(u, dtype=np.float32)
    _load().vgs_fill_query(seed, stream, start, count, d, _ptr(u), _ptr(out))
    return out


def choose(seed, stream, lo, hi, m, value, flags: np.ndarray) -> None:
    assert flags.dtype == np.uint8 and flags.flags.c_contiguous
    if _load().vgs_choose(seed, stream, lo, hi, m, value, _ptr(flags)) != 0:
        raise ValueError("bad choose() arguments")


def uniform_int(seed, stream, idx, lo, hi) -> int:
    return int(_load().vgs_uniform_int(seed, stream, idx, lo, hi))


# ---------------------------------------------------------------- workloads
@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    gamma: int
    k: int
    n: int | None                 # fixed prefix length, or None when ragged
    ragged: tuple | None = None   # (lo, hi) inclusive, per sequence
    layers: int = 1
    scheme: str = "iid"           # "iid" | "heavy"
    heavy_frac: float = 0.0
    sinks: int = 0
    u_per_seq: bool = False
    select_rows: str = "c2"       # rows the selection uses: "c2" or "all"
    extra_rows: str | None = None  # second aggregation in the same pass, or None
    seed: int = 1000
    description: str = field(default="", compare=False)

    @property
    def R(self) -> int:
        return self.gamma + 1

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def rows(self, which: str) -> list[int]:
        """Verify rows a mask aggregates: Collect-2-Query = first draft row and bonus row."""
        if which == "c2":
            return sorted({0, self.gamma})
        if which == "all":
            return list(range(self.R))
        raise ValueError(which)

    def row_mask(self, which: str | None) -> int:
        if which is None:
            return 0
        m = 0
        for t in self.rows(which):
            m |= 1 << t
        return m

    def lengths(self, layer: int = 0) -> np.ndarray:
        """Prefix length n_b of every sequence (the same for every layer)."""
        if self.ragged is None:
            return np.full(self.B, self.n, dtype=np.int64)
        lo, hi = self.ragged
        return np.array([uniform_int(self.seed, stream_id(T_LEN, 0, 0), b, lo, hi)
                         for b in range(self.B)], dtype=np.int64)

    def max_len(self) -> int:
        return int(self.lengths().max())

    # -- per-sequence pieces ------------------------------------------------
    def direction(self, layer: int, b: int) -> np.ndarray | None:
        if self.scheme == "iid":
            return None
        return unit_vector(self.seed, stream_id(T_U, layer, b if self.u_per_seq else 0), self.d)

    def key_kinds(self, layer: int, b: int, n: int) -> np.ndarray | None:
        """0 = N(0,1) key, 1 = heavy hitter 3u + N(0, 0.5^2), 2 = sink 4u."""
        if self.scheme == "iid":
            return None
        kind = np.zeros(n, dtype=np.uint8)
        s = min(self.sinks, n)
        kind[:s] = 2
        m = int(np.floor(self.heavy_frac * n))
        m = min(m, n - s)
        choose(self.seed, stream_id(T_HEAVY, layer, b), s, n, m, 1, kind)
        return kind

    def prefix_k(self, layer: int, b: int, pos0: int = 0, npos: int | None = None) -> np.ndarray:
        n = int(self.lengths()[b])
        npos = n - pos0 if npos is None else npos
        kind = self.key_kinds(layer, b, n)
        kk = None if kind is None else kind[pos0:pos0 + npos]
        return keys_bf16(self.seed, stream_id(T_K, layer, b), pos0, npos, self.Hkv, self.d, kk,
                         self.direction(layer, b))

    def prefix_v(self, layer: int, b: int, pos0: int = 0, npos: int | None = None) -> np.ndarray:
        n = int(self.lengths()[b])
        npos = n - pos0 if npos is None else npos
        return keys_bf16(self.seed, stream_id(T_V, layer, b), pos0, npos, self.Hkv, self.d)

    def verify_q(self, layer: int, b: int) -> np.ndarray:
        """[R][H_q][d] verify queries: rows 0..gamma-1 draft tokens, row gamma the bonus."""
        c = self.R * self.Hq * self.d
        return query_bf16(self.seed, stream_id(T_QV, layer, b), c, self.d,
                          self.direction(layer, b)).reshape(self.R, self.Hq, self.d)

    def verify_kv_new(self, layer: int, b: int) -> tuple[np.ndarray, np.ndarray]:
        c = self.R * self.Hkv * self.d
        kn = normal_bf16(self.seed, stream_id(T_KNEW, layer, b), c)
        vn = normal_bf16(self.seed, stream_id(T_VNEW, layer, b), c)
        shp = (self.R, self.Hkv, self.d)
        return kn.reshape(shp), vn.reshape(shp)

    def draft_q(self, layer: int, b: int) -> np.ndarray:
        """[gamma][H_q][d] draft-step queries."""
        c = self.gamma * self.Hq * self.d
        return query_bf16(self.seed, stream_id(T_QD, layer, b), c, self.d,
                          self.direction(layer, b)).reshape(self.gamma, self.Hq, self.d)

    def draft_kv(self, layer: int, b: int) -> tuple[np.ndarray, np.ndarray]:
        c = self.gamma * self.Hkv * self.d
        kd = normal_bf16(self.seed, stream_id(T_KD, layer, b), c)
        vd = normal_bf16(self.seed, stream_id(T_VD, layer, b), c)
        shp = (self.gamma, self.Hkv, self.d)
        return kd.reshape(shp), vd.reshape(shp)

    # -- the whole layer, laid out as a token-granular slot pool ------------
    def slot_layout(self) -> tuple[np.ndarray, int]:
        """seq_offset[b] (first slot of sequence b) and the pool's slot count.

        Each sequence reserves n_b + gamma + 1 slots (prefix, then the verify rows,
        which the draft tokens later reuse), rounded up to 16 slots."""
        n = self.lengths()
        cap = ((n + self.R + 15) // 16) * 16
        off = np.zeros(self.B, dtype=np.int64)
        off[1:] = np.cumsum(cap)[:-1]
        return off, int(cap.sum())

    def layer_pool(self, layer: int = 0) -> dict:
        """Everything one layer needs, as host arrays (bf16 as uint16)."""
        n = self.lengths()
        off, slots = self.slot_layout()
        K = np.zeros((slots, self.Hkv, self.d), dtype=np.uint16)
        V = np.zeros((slots, self.Hkv, self.d), dtype=np.uint16)
        for b in range(self.B):
            o, nb = int(off[b]), int(n[b])
            K[o:o + nb] = self.prefix_k(layer, b)
            V[o:o + nb] = self.prefix_v(layer, b)
        qv = np.stack([self.verify_q(layer, b) for b in range(self.B)])
        kvn = [self.verify_kv_new(layer, b) for b in range(self.B)]
        qd = np.stack([self.draft_q(layer, b) for b in range(self.B)], axis=1)
        kvd = [self.draft_kv(layer, b) for b in range(self.B)]
        return dict(
            K=K, V=V, seq_offset=off, prefix_len=n.astype(np.int32), slots=slots,
            q_verify=qv,                                          # [B][R][Hq][d]
            k_new=np.stack([a for a, _ in kvn]),                  # [B][R][Hkv][d]
            v_new=np.stack([c for _, c in kvn]),
            q_draft=qd,                                           # [gamma][B][Hq][d]
            k_draft=np.stack([a for a, _ in kvd], axis=1),        # [gamma][B][Hkv][d]
            v_draft=np.stack([c for _, c in kvd], axis=1),
        )


WORKLOADS = {
    "tiny": Workload("tiny", B=1, Hq=8, Hkv=2, d=64, gamma=3, k=64, n=512, seed=1001,
                     description="tiny correctness case, i.i.d. N(0,1)"),
    "llama8b": Workload("llama8b", B=1, Hq=32, Hkv=8, d=128, gamma=7, k=2048, n=32768,
                        scheme="heavy", heavy_frac=0.02, seed=1002,
                        description="Llama-3-8B-shaped layer, n=32768, 2% heavy hitters"),
    "batched": Workload("batched", B=16, Hq=32, Hkv=8, d=128, gamma=7, k=1024, n=16384,
                        scheme="heavy", heavy_frac=0.02, u_per_seq=True, select_rows="all",
                        extra_rows="c2", seed=1003,
                        description="16 sequences x 16384, all-rows selection + C2 overlap"),
    "long70b": Workload("long70b", B=1, Hq=64, Hkv=8, d=128, gamma=5, k=4096, n=131072,
                        scheme="heavy", heavy_frac=0.01, sinks=16, seed=1004,
                        description="70B-shaped layer, n=131072, 1% heavy hitters + 16 sinks"),
    "loop32": Workload("loop32", B=8, Hq=32, Hkv=8, d=128, gamma=6, k=2048, n=None,
                       ragged=(4096, 65536), layers=32, scheme="heavy", heavy_frac=0.02,
                       u_per_seq=True, seed=1005,
                       description="32 layers, 8 ragged sequences n~U[4096,65536]"),
}


# ---------------------------------------------------------------- paged layout
def to_paged(w: "Workload", pool: dict, page_size: int, seed: int = 0) -> dict:
    """The same layer laid out as a paged cache: every sequence's tokens (prefix plus the
    gamma+1 verify rows) in pages of page_size slots, the pages of all sequences spread
    over the pool by a seeded permutation (seed None: in order, an identity table).  Returns the pool dict with K and V
    re-arranged, page_table int32 [B][pages_per_seq] and page_size; the logical content
    is unchanged (layout only, no attention arithmetic)."""
    n = pool["prefix_len"].astype(np.int64)
    need = (n + w.R + page_size - 1) // page_size                  # pages per sequence
    pages_per_seq = int(need.max())
    total = int(need.sum())
    perm = np.arange(total) if seed is None else np.random.default_rng(seed).permutation(total)
    table = np.full((w.B, pages_per_seq), -1, dtype=np.int32)
    K = np.zeros((total * page_size,) + pool["K"].shape[1:], dtype=np.uint16)
    V = np.zeros_like(K)
    k = 0
    for b in range(w.B):
        o = int(pool["seq_offset"][b])
        cap = int(pool["seq_offset"][b + 1]) - o if b + 1 < w.B else pool["K"].shape[0] - o
        for j in range(int(need[b])):
            pg = int(perm[k])
            k += 1
            table[b, j] = pg
            lo, hi = j * page_size, min((j + 1) * page_size, cap)
            if lo < hi:
                K[pg * page_size:pg * page_size + hi - lo] = pool["K"][o + lo:o + hi]
                V[pg * page_size:pg * page_size + hi - lo] = pool["V"][o + lo:o + hi]
    out = dict(pool)
    out.update(K=K, V=V, page_table=table, page_size=page_size, slots=total * page_size)
    return out


# ---------------------------------------------------------------- acceptance inputs
def accept_inputs(B: int, gamma: int, V: int, seed: int, scale: float = 3.0, noise: float = 1.0) -> dict:
    """Synthetic inputs of the acceptance step (fp32 logits, as a model's output head
    gives them): target logits p [B][gamma+1][V] = scale * N(0,1); draft logits
    q [B][gamma][V] = p[:, :gamma] + noise * N(0,1) (a draft close to the target); draft
    tokens x [B][gamma] drawn from the draft's distribution by the Gumbel-max trick
    (argmax of q plus Gumbel noise, which samples softmax(q) without computing it);
    uniforms u [B][gamma] and u_res [B] in [0, 1).  numpy's seeded generator."""
    r = np.random.default_rng(seed)
    p = (scale * r.standard_normal((B, gamma + 1, V))).astype(np.float32)
    q = (p[:, :gamma] + noise * r.standard_normal((B, gamma, V))).astype(np.float32)
    gumbel = -np.log(-np.log(r.uniform(1e-12, 1.0, size=(B, gamma, V))))
    x = np.argmax(q.astype(np.float64) + gumbel, axis=-1).astype(np.int32) if gamma else np.zeros((B, 0), np.int32)
    u = r.uniform(0.0, 1.0, size=(B, gamma)).astype(np.float32)
    u_res = r.uniform(0.0, 1.0, size=B).astype(np.float32)
    return dict(p_logits=p, q_logits=q, x=x, u=u, u_res=u_res)


def scaled(w: Workload, **kw) -> Workload:
    """A copy of a workload with some fields replaced (small parity cases)."""
    from dataclasses import replace
    return replace(w, **kw)
