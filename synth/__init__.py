"""Seeded synthetic inputs for the DFlash2 draft tail (shared by the oracle and the CUDA path).

Holds none of the draft tail's arithmetic: only the counter-based generator
(Philox4x32-10, Salmon et al., SC'11), the Box-Muller normals built from it, and
the input recipes (shapes, scales, RMS normalisation of the hidden rows, planted
peaks) for the five workloads. The planted peaks are stored data: the planted tokens'
lm_head rows are moved by deltas that a committed script computed once from the CPU
oracle's conv output (``tests/golden/make_planted_rows.py``); this module only draws
which slots are planted with which token and adds the stored deltas. The C core is ``synth.c``; this module compiles it
with the host C compiler on first use and loads it with ctypes.

Tensor ids (the second Philox key word) are fixed per tensor so the order in
which tensors are generated does not matter.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

TID_HIDDEN = 1
TID_LM_HEAD = 2
TID_U = 3
TID_V = 4
TID_CONV_W = 16  # + layer index
TID_ANCHOR = 32
TID_ANCHOR_DUP = 33
TID_PLANT_ID = 34
TID_PLANT_ON = 35
TID_GATE_W = 36


def build(force: bool = False) -> str:
    """Compile ``libsynth.so`` next to its source (host gcc, -O2, pthreads)."""
    with _lock:
        if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        u32, u64, i32, dbl = ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int, ctypes.c_double
        vp = ctypes.c_void_p
        lib.synth_philox4x32_10.argtypes = [vp, vp, vp]
        lib.synth_f64_to_bf16.argtypes = [dbl]
        lib.synth_f64_to_bf16.restype = ctypes.c_uint16
        for name in ("synth_normal_bf16", "synth_normal_f32", "synth_normal_f64"):
            getattr(lib, name).argtypes = [u32, u32, dbl, u64, vp, i32]
        lib.synth_uniform_f64.argtypes = [u32, u32, u64, vp]
        lib.synth_uniform_int.argtypes = [u32, u32, u64, ctypes.c_int64, vp]
        lib.synth_round_bf16.argtypes = [vp, u64, vp]
        _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def philox4x32_10(ctr, key) -> tuple:
    """One Philox4x32-10 block: 4 counter words, 2 key words -> 4 output words."""
    lib = _load()
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    o = np.zeros(4, dtype=np.uint32)
    lib.synth_philox4x32_10(c.ctypes.data, k.ctypes.data, o.ctypes.data)
    return tuple(int(x) for x in o)


def normal(seed: int, tid: int, shape, std: float, kind: str = "bf16") -> np.ndarray:
    """N(0, std^2) samples. kind: 'bf16' (uint16 bit patterns), 'f32' or 'f64'."""
    lib = _load()
    count = int(np.prod(shape))
    dt = {"bf16": np.uint16, "f32": np.float32, "f64": np.float64}[kind]
    out = np.empty(count, dtype=dt)
    fn = {"bf16": lib.synth_normal_bf16, "f32": lib.synth_normal_f32, "f64": lib.synth_normal_f64}[kind]
    if count:
        fn(seed, tid, float(std), count, out.ctypes.data, _threads())
    return out.reshape(shape)


def uniform(seed: int, tid: int, count: int) -> np.ndarray:
    lib = _load()
    out = np.empty(count, dtype=np.float64)
    if count:
        lib.synth_uniform_f64(seed, tid, count, out.ctypes.data)
    return out


def uniform_int(seed: int, tid: int, count: int, n: int) -> np.ndarray:
    lib = _load()
    out = np.empty(count, dtype=np.int64)
    if count:
        lib.synth_uniform_int(seed, tid, count, int(n), out.ctypes.data)
    return out


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round doubles to bf16 bit patterns (nearest, ties to even, no double rounding)."""
    lib = _load()
    a = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    if a.size:
        lib.synth_round_bf16(a.ctypes.data, a.size, out.ctypes.data)
    return out


def bf16_bits_to_f32(u16: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (a storage conversion)."""
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# Workload recipes
# ---------------------------------------------------------------------------

@dataclass
class Shape:
    batch: int
    block: int
    hidden: int
    vocab: int
    top_k: int
    rank: int
    group_size: int = 16
    kernel_size: int = 2
    layers: int = 5
    dtype: str = "bf16"  # 'bf16' or 'f32'
    taps: str = "softmax"  # 'softmax' (default) or 'raw'
    gate: bool = False     # context gate H(h_t) in the transition scores
    first_slot: int = 0    # 1: row 0 of each block is the anchor's position, slots are rows 1..block-1

    @property
    def rows(self) -> int:
        return self.batch * self.block

    @property
    def taps_per_layer(self) -> int:
        return 2 * (self.hidden // self.group_size)


@dataclass
class Recipe:
    """How a workload's tensors are drawn. std values are standard deviations."""
    seed: int
    shape: Shape
    hidden_std: float = 1.0
    rms_normalise: bool = False
    lm_head_std: float = 0.02
    uv_std: float = 0.05
    conv_std: float = 0.02
    gate_std: float = 0.0  # 0: 1 / sqrt(hidden), so a gate entry of a unit-rms row is about N(0, 1)
    plant: str = "none"  # 'none', 'all' (every slot, 1 % left unplanted), 'even_rows' (slots t even)
    anchor_dup_frac: float = 0.0
    name: str = ""
    extra: dict = field(default_factory=dict)


# Planted peaks: a planted slot's token gets top-1 probability PLANT_MASS at that slot (its
# logit set to the log-sum-exp of the slot's other logits plus log(PLANT_MASS / (1 - PLANT_MASS)))
# through a change of that token's lm_head row that leaves the logits of the sequence's other
# slots unchanged; the deltas are stored per workload under tests/golden.
PLANT_MASS = 0.85
PLANT_SKIP = 0.01  # 'all': the share of slots left unplanted
GOLDEN_DIR = os.path.join(os.path.dirname(_HERE), "tests", "golden")


def planted_rows_path(rc: "Recipe") -> str:
    return os.path.join(GOLDEN_DIR, f"planted_rows_{rc.name}.npz")


def recipe(config: int) -> Recipe:
    """The five workloads: a tiny fp32 instance and four page-shape instances."""
    page = dict(hidden=5120, vocab=248320, top_k=16, rank=256, group_size=16, kernel_size=2, layers=5)
    if config == 1:
        sh = Shape(batch=1, block=4, hidden=256, vocab=4096, top_k=4, rank=32, layers=1, dtype="f32")
        return Recipe(seed=0, shape=sh, hidden_std=1.0, lm_head_std=1.0 / 16.0, uv_std=0.1, conv_std=0.05,
                      name="tiny_fp32_b1_t4_h256_v4096_k4_r32")
    if config == 2:
        return Recipe(seed=1, shape=Shape(batch=1, block=8, **page), rms_normalise=True,
                      name="page_b1_t8_h5120_v248320_k16_r256")
    if config == 3:
        return Recipe(seed=2, shape=Shape(batch=8, block=8, **page), rms_normalise=True,
                      plant="all", name="page_b8_t8_planted")
    if config == 4:
        return Recipe(seed=3, shape=Shape(batch=32, block=8, **page), rms_normalise=True,
                      anchor_dup_frac=0.25, name="page_b32_t8_dup_anchors")
    if config == 5:
        return Recipe(seed=4, shape=Shape(batch=64, block=16, **page), rms_normalise=True,
                      plant="even_rows", name="stress_b64_t16_half_planted")
    raise ValueError(f"unknown workload {config}")


def scaled_recipe(base: Recipe, **shape_overrides) -> Recipe:
    """Same distributions, other sizes (small parity cases)."""
    sh = Shape(**{**base.shape.__dict__, **shape_overrides})
    return Recipe(**{**base.__dict__, "shape": sh})


def planted_slots(rc: Recipe) -> np.ndarray:
    """[B, T] int32: the token planted at each slot, -1 where none. 'all': every slot but about
    PLANT_SKIP of them; 'even_rows': the slots t even. Tokens are distinct across the workload
    (a repeat moves to the next free id)."""
    sh = rc.shape
    B, T, Vv = sh.batch, sh.block, sh.vocab
    out = np.full((B, T), -1, dtype=np.int32)
    if rc.plant == "none":
        return out
    ids = uniform_int(rc.seed, TID_PLANT_ID, B * T, Vv).reshape(B, T)
    on_u = uniform(rc.seed, TID_PLANT_ON, B * T).reshape(B, T)
    used = set()
    for b in range(B):
        for t in range(T):
            if rc.plant == "all" and on_u[b, t] >= 1.0 - PLANT_SKIP:
                continue
            if rc.plant == "even_rows" and t % 2 == 1:
                continue
            if len(used) >= Vv:
                raise ValueError(f"more planted slots than the {Vv} vocabulary ids")
            p = int(ids[b, t])
            while p in used:
                p = (p + 1) % Vv
            used.add(p)
            out[b, t] = p
    return out


def apply_planted_rows(rc: Recipe, lm_head: np.ndarray, planted: np.ndarray) -> None:
    """Add the stored deltas to the planted tokens' lm_head rows (bf16, in place): row p becomes
    bf16(row p + step * code), the codes stored as int8 values -127..127, step the row's step."""
    path = planted_rows_path(rc)
    if not os.path.exists(path):
        raise FileNotFoundError(f"{path} is missing; tests/golden/make_planted_rows.py writes it")
    st = np.load(path)
    ids = planted[planted >= 0]
    if not np.array_equal(st["ids"], ids):
        raise ValueError(f"{path} was written for other planted slots")
    q = st["q"].astype(np.float64)
    rows = bf16_bits_to_f32(lm_head[ids]).astype(np.float64) + q * st["step"][:, None]
    lm_head[ids] = f64_to_bf16(rows)


def make_inputs(rc: Recipe, with_lm_head: bool = True, apply_planting: bool = True) -> dict:
    """Generate every input tensor of one workload.

    Returns numpy arrays: ``hidden`` [B,T,H], ``lm_head`` [V,H], ``U``/``V`` [V,R],
    ``conv_w`` [NL,P,H], ``gate_w`` [R,H] (bf16 bit patterns as uint16, or float32 for
    dtype f32) and
    ``anchor`` [B] int32, plus ``planted`` [B,T] int32 (-1 where a slot is not planted).
    With ``apply_planting`` False the planted tokens' rows are left as drawn (the state the
    stored deltas were computed from).
    """
    sh = rc.shape
    B, T, H, Vv, R = sh.batch, sh.block, sh.hidden, sh.vocab, sh.rank
    NL, P = sh.layers, sh.taps_per_layer
    kind = "bf16" if sh.dtype == "bf16" else "f32"
    s = rc.seed
    out = {}
    out["lm_head"] = normal(s, TID_LM_HEAD, (Vv, H), rc.lm_head_std, kind) if with_lm_head else None
    out["U"] = normal(s, TID_U, (Vv, R), rc.uv_std, kind)
    out["V"] = normal(s, TID_V, (Vv, R), rc.uv_std, kind)
    gate_std = rc.gate_std if rc.gate_std > 0 else 1.0 / np.sqrt(H)
    out["gate_w"] = normal(s, TID_GATE_W, (R, H), gate_std, kind)
    out["conv_w"] = np.stack([normal(s, TID_CONV_W + l, (P, H), rc.conv_std, kind) for l in range(NL)]) \
        if NL > 0 else np.zeros((0, P, H), dtype=np.uint16 if kind == "bf16" else np.float32)

    anchor = uniform_int(s, TID_ANCHOR, B, Vv)
    if rc.anchor_dup_frac > 0 and B > 1:
        n_dup = int(round(B * rc.anchor_dup_frac))
        n_src = B - n_dup
        pick = uniform_int(s, TID_ANCHOR_DUP, n_dup, n_src)
        anchor[n_src:] = anchor[pick]
    out["anchor"] = anchor.astype(np.int32)

    h = normal(s, TID_HIDDEN, (B, T, H), rc.hidden_std, "f64")
    if rc.rms_normalise:
        h = h / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + 1e-6)
    out["hidden"] = f64_to_bf16(h) if kind == "bf16" else h.astype(np.float32)
    planted = planted_slots(rc)
    if rc.plant != "none" and apply_planting:
        if out["lm_head"] is None:
            raise ValueError("planting needs the lm_head rows")
        apply_planted_rows(rc, out["lm_head"], planted)
    out["planted"] = planted
    return out
