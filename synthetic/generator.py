"""Counter-based seeded generator for the VLA workloads.

Random numbers
--------------
Every value is a pure function of ``(seed, stream, index)``:

* ``key = mix64(seed * 0xD1B54A32D192ED03 + stream * 0x9E3779B97F4A7C15 + 1)``
* ``bits(i) = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)`` (mod 2**64)

where ``mix64`` is the SplitMix64 output function (Steele, Lea, Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014):
``z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27; z *= 0x94D049BB133111EB;
z ^= z >> 31``.  A uniform double is ``(bits >> 11) * 2**-53`` in [0, 1).
Standard normals come in pairs from the Box-Muller transform in fp64:
element ``2j`` is ``sqrt(-2 ln(1 - U_{2j})) cos(2 pi U_{2j+1})`` and element
``2j+1`` the same with ``sin``.

Precision
---------
fp32 inputs are the fp64 normals rounded to nearest fp32.  bf16 inputs are
those fp32 values rounded to nearest-even bf16; they are carried as raw
``uint16`` bit patterns because numpy has no bf16 type.  Both the oracle and
the GPU path receive the same bits (the oracle upcasts them exactly).

Workloads
---------
``CONFIGS`` holds the five synthetic configurations of the VLA forward
recurrence (key/value/query/penalty-direction tensors laid out
``[B, H, T, d]``).  Shapes and distributions follow the workloads stated for
this recurrence; the key-value recall stream (config 5) stands in for the
multi-query associative recall task of "Variational Linear Attention: Stable
Associative Memory for Long-Context Transformers", section 4, whose data set
is not available.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

_GOLD = np.uint64(0x9E3779B97F4A7C15)
_SEEDMUL = np.uint64(0xD1B54A32D192ED03)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# stream ids of the four per-token input tensors
STREAM_Q, STREAM_K, STREAM_V, STREAM_U = 0, 1, 2, 3


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * _M1
    z = z ^ (z >> np.uint64(27))
    z = z * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        x = (np.uint64(seed & 0xFFFFFFFFFFFFFFFF) * _SEEDMUL
             + np.uint64(stream & 0xFFFFFFFFFFFFFFFF) * _GOLD + np.uint64(1))
        return _mix64(np.array([x], dtype=np.uint64))[0]


def uniforms(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Uniform doubles in [0,1) for counter indices [start, start+count)."""
    key = _key(seed, stream)
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        bits = _mix64(key + idx * _GOLD)
    return (bits >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def normals(seed: int, stream: int, count: int, start: int = 0,
            block: int = 1 << 22) -> np.ndarray:
    """``count`` standard normals (fp64), element i uses counters 2*(i//2), 2*(i//2)+1.

    ``start`` must be even.  Generated in blocks to bound temporary memory.
    """
    assert start % 2 == 0
    out = np.empty(count, dtype=np.float64)
    npairs = (count + 1) // 2
    p0 = 0
    while p0 < npairs:
        p1 = min(npairs, p0 + block)
        uu = uniforms(seed, stream, start + 2 * p0, 2 * (p1 - p0))
        u1 = 1.0 - uu[0::2]
        u2 = uu[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        th = (2.0 * np.pi) * u2
        seg = np.empty(2 * (p1 - p0), dtype=np.float64)
        seg[0::2] = r * np.cos(th)
        seg[1::2] = r * np.sin(th)
        lo = 2 * p0
        hi = min(count, 2 * p1)
        out[lo:hi] = seg[: hi - lo]
        p0 = p1
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to nearest-even bf16; returns the uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    # NaN stays NaN (quiet); none are generated here.
    rnd = np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))
    return ((b + rnd) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


@dataclasses.dataclass
class VLAInputs:
    """One batch of inputs.  Arrays are ``[B, H, T, d]``.

    For ``dtype == "bf16"`` the arrays are ``uint16`` bf16 bit patterns,
    for ``"f32"`` they are ``float32``.
    """

    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    u: np.ndarray
    dtype: str
    lambda0: float
    name: str = ""
    # key-value recall streams only: [B, H, n, d] fp64 keys (unit) and values
    keys: Optional[np.ndarray] = None
    values: Optional[np.ndarray] = None

    @property
    def shape(self):
        return self.q.shape

    def as_f64(self, name: str) -> np.ndarray:
        """Exact fp64 copy of one input tensor."""
        a = getattr(self, name)
        if self.dtype == "bf16":
            return bf16_bits_to_f32(a).astype(np.float64)
        return a.astype(np.float64)

    def as_f32(self, name: str) -> np.ndarray:
        a = getattr(self, name)
        if self.dtype == "bf16":
            return bf16_bits_to_f32(a)
        return a.astype(np.float32)

    def slice_heads(self, b: slice, h: slice) -> "VLAInputs":
        return dataclasses.replace(
            self,
            q=np.ascontiguousarray(self.q[b, h]), k=np.ascontiguousarray(self.k[b, h]),
            v=np.ascontiguousarray(self.v[b, h]), u=np.ascontiguousarray(self.u[b, h]),
            keys=None if self.keys is None else self.keys[b, h],
            values=None if self.values is None else self.values[b, h],
        )


def _round(x64: np.ndarray, dtype: str) -> np.ndarray:
    x32 = x64.astype(np.float32)
    if dtype == "f32":
        return x32
    if dtype == "bf16":
        return f32_to_bf16_bits(x32)
    raise ValueError(dtype)


def make_inputs(B: int, H: int, T: int, d: int, dtype: str = "f32", seed: int = 0,
                lambda0: float = 1.0, u_scale: float = 1.0,
                unit_keys: bool = False, name: str = "") -> VLAInputs:
    """i.i.d. N(0,1) q, k, v and N(0, u_scale^2) u, each from its own stream.

    ``unit_keys`` pre-normalises every key to unit length in fp64 before
    rounding (the tiny fp32 configuration states its keys that way).
    """
    n = B * H * T * d
    shp = (B, H, T, d)
    out = {}
    for nm, st in (("q", STREAM_Q), ("k", STREAM_K), ("v", STREAM_V), ("u", STREAM_U)):
        x = normals(seed, st, n).reshape(shp)
        if nm == "u" and u_scale != 1.0:
            x = x * u_scale
        if nm == "k" and unit_keys:
            x = x / np.linalg.norm(x, axis=-1, keepdims=True)
        out[nm] = _round(x, dtype)
    return VLAInputs(out["q"], out["k"], out["v"], out["u"], dtype, float(lambda0), name=name)


def make_recall_stream(B: int, H: int, T: int, d: int, n_pairs: int, seed: int = 5,
                       dtype: str = "f32", lambda0: float = 1.0,
                       distractor_std: float = 0.1, name: str = "") -> VLAInputs:
    """Synthetic key-value recall streams.

    Per (b, h): ``n_pairs`` keys, random orthonormal when ``n_pairs <= d``
    (Q factor of a seeded Gaussian d x n matrix) else random unit vectors,
    values ~ N(0,1).  Token 2i and 2i+1 write pair i (k = key_i, v = value_i,
    u = key_i).  Tokens 2n .. T-n-1 are distractors with q, k, v, u ~
    N(0, distractor_std^2).  The last n tokens query pair i with q = key_i
    (their k, v, u are distractors too).  q of the write tokens is distractor
    noise.  Requires T >= 3 * n_pairs.
    """
    if T < 3 * n_pairs:
        raise ValueError("T must be >= 3 * n_pairs")
    shp = (B, H, T, d)
    cnt = B * H * T * d
    q = normals(seed, STREAM_Q, cnt).reshape(shp) * distractor_std
    k = normals(seed, STREAM_K, cnt).reshape(shp) * distractor_std
    v = normals(seed, STREAM_V, cnt).reshape(shp) * distractor_std
    u = normals(seed, STREAM_U, cnt).reshape(shp) * distractor_std
    g = normals(seed, 16, B * H * d * n_pairs).reshape(B, H, d, n_pairs)
    vals = normals(seed, 17, B * H * n_pairs * d).reshape(B, H, n_pairs, d)
    keys = np.empty((B, H, n_pairs, d))
    for b in range(B):
        for h in range(H):
            if n_pairs <= d:
                qm, _ = np.linalg.qr(g[b, h])
                keys[b, h] = qm.T
            else:
                keys[b, h] = (g[b, h] / np.linalg.norm(g[b, h], axis=0, keepdims=True)).T
    # keys and values are rounded to the I/O precision first so that the
    # recall targets are exactly what the recurrence receives.
    if dtype == "bf16":
        keys = bf16_bits_to_f32(_round(keys, dtype)).astype(np.float64)
        vals = bf16_bits_to_f32(_round(vals, dtype)).astype(np.float64)
    else:
        keys = keys.astype(np.float32).astype(np.float64)
        vals = vals.astype(np.float32).astype(np.float64)
    for i in range(n_pairs):
        for t in (2 * i, 2 * i + 1):
            k[:, :, t] = keys[:, :, i]
            v[:, :, t] = vals[:, :, i]
            u[:, :, t] = keys[:, :, i]
        q[:, :, T - n_pairs + i] = keys[:, :, i]
    return VLAInputs(_round(q, dtype), _round(k, dtype), _round(v, dtype), _round(u, dtype),
                     dtype, float(lambda0), name=name, keys=keys, values=vals)


# The five workloads.  Each entry: constructor kwargs for make_inputs /
# make_recall_stream.  "tiny" is the small fp32 case the oracle finishes in
# well under a second; "heads32" is B=4 H=8 T=4096 d=64 bf16; "long" is the
# long stream B=1 H=16 T=65536 d=64 bf16 with u scaled by 0.5; "batched" is
# B=32 H=16 T=2048 d=128 bf16 with lambda0=0.5; "recall" is the key-value
# recall streams B=256 H=4 T=512 d=32 fp32 with n in {8, 24, 48}; "decode" is
# one token per call for B=32 H=64 d=64 bf16 with the state kept in HBM.
CONFIGS = {
    "tiny": dict(kind="iid", B=1, H=1, T=256, d=32, dtype="f32", seed=0, lambda0=1.0,
                 unit_keys=True),
    "heads32": dict(kind="iid", B=4, H=8, T=4096, d=64, dtype="bf16", seed=2, lambda0=1.0),
    "long": dict(kind="iid", B=1, H=16, T=65536, d=64, dtype="bf16", seed=3, lambda0=1.0,
                 u_scale=0.5),
    "batched": dict(kind="iid", B=32, H=16, T=2048, d=128, dtype="bf16", seed=4,
                    lambda0=0.5),
    "recall8": dict(kind="recall", B=256, H=4, T=512, d=32, n_pairs=8, dtype="f32", seed=5),
    "recall24": dict(kind="recall", B=256, H=4, T=512, d=32, n_pairs=24, dtype="f32", seed=5),
    "recall48": dict(kind="recall", B=256, H=4, T=512, d=32, n_pairs=48, dtype="f32", seed=5),
    # streaming decode step: one token per call for 2048 (b, h) units
    "decode": dict(kind="iid", B=32, H=64, T=1, d=64, dtype="bf16", seed=6, lambda0=1.0),
}


def make_config(name: str, **override) -> VLAInputs:
    """Build one of ``CONFIGS`` (keyword overrides allowed, e.g. a smaller T or B)."""
    spec = dict(CONFIGS[name])
    spec.update(override)
    kind = spec.pop("kind")
    if kind == "iid":
        return make_inputs(name=name, **spec)
    return make_recall_stream(name=name, **spec)
