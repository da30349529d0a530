"""The tensor-core chunked path (VLA_KERNEL_CHUNK_TC: d_h = 64, bf16 I/O,
block-Woodbury gates and UT-transform state passes) against the fp64 oracle
on the inputs where the method has its special cases:

- keys of norm zero or below eps (the max(|k|, eps) guard of the unit key,
  section 2.3), at sub-block and chunk boundaries;
- u = 0 (no penalty update: A stays I / lambda0 and the gate is the key, the
  delta rule), u scaled by 10 and by 0.01 (capacitance matrices I + U^T A U
  from badly to very well conditioned);
- lambda0 = 0.01 and 100 (A_0 = 100 I and 0.01 I);
- the key-value recall streams at d_h = 64 (orthonormal keys, u = k_hat, each
  pair written twice: gates equal to the keys, c_t = 1, repeated columns in
  the sub-block systems), with the recall error |S k_i - v_i| from the GPU's
  state against the oracle's.

Every case spans several chunks and a ragged last sub-block.  Bar: relative
Frobenius error <= 5e-3 per output (bf16 I/O, fp32 state)."""

import numpy as np
import pytest

import rls_associative_memory_gb300 as vla
from synthetic import make_inputs, make_recall_stream
from vla_testutil import TOL, compare, oracle_ref, run_gpu, to_device

pytestmark = pytest.mark.gpu

TC = vla.VLA_KERNEL_CHUNK_TC
CHUNKS = [128, 192, 0]  # two and three sub-blocks per chunk (ragged), and the default


def _zero_keys(x, positions, scale=0.0):
    """Keys at `positions` replaced by 0 (scale 0) or by scale * the key
    (bf16 bits of the scaled value), in every (b, h) unit."""
    from synthetic.generator import f32_to_bf16_bits
    k = x.as_f32("k")
    for t in positions:
        k[:, :, t, :] *= scale
    x.k = f32_to_bf16_bits(k) if x.dtype == "bf16" else k
    return x


@pytest.mark.parametrize("chunk", CHUNKS)
def test_zero_and_tiny_keys(chunk):
    x = make_inputs(1, 4, 1000, 64, "bf16", seed=61, u_scale=0.5)
    # sub-block boundaries 63 | 64, chunk boundaries 127 | 128 and 191 | 192, the ends
    x = _zero_keys(x, [0, 1, 63, 64, 127, 128, 191, 192, 500, 999], 0.0)
    # keys far below eps = 1e-6 in norm (k_hat = k / eps is then not a unit vector)
    x = _zero_keys(x, [2, 65, 129, 640, 998], 1e-8)
    compare(run_gpu(x, TC, chunk=chunk), oracle_ref(x), "bf16")


@pytest.mark.parametrize("chunk", CHUNKS)
@pytest.mark.parametrize("u_scale", [0.0, 0.01, 10.0], ids=["u0", "u0.01", "u10"])
def test_penalty_scale(u_scale, chunk):
    x = make_inputs(1, 4, 1000, 64, "bf16", seed=62, u_scale=u_scale)
    ref = oracle_ref(x)
    got = run_gpu(x, TC, chunk=chunk)
    compare(got, ref, "bf16")
    if u_scale == 0.0:
        # no penalty update: A_T = A_0 (= I here) up to the rounding of the restarts
        assert np.max(np.abs(got["A_T"] - np.eye(64))) <= 1e-6


@pytest.mark.parametrize("chunk", CHUNKS)
@pytest.mark.parametrize("lambda0", [0.01, 100.0])
def test_lambda0_extremes(lambda0, chunk):
    x = make_inputs(1, 4, 1000, 64, "bf16", seed=63, u_scale=0.5, lambda0=lambda0)
    compare(run_gpu(x, TC, chunk=chunk), oracle_ref(x), "bf16")


def _recall_errors(S, keys, vals):
    return np.linalg.norm(np.einsum("...ij,...nj->...ni", S, keys) - vals, axis=-1)


@pytest.mark.parametrize("n_pairs", [24, 64])
@pytest.mark.parametrize("chunk", [128, 0])
def test_recall_streams_d64(n_pairs, chunk):
    x = make_recall_stream(2, 2, 1024, 64, n_pairs, seed=64, dtype="bf16")
    ref = oracle_ref(x)
    got = run_gpu(x, TC, chunk=chunk)
    compare(got, ref, "bf16")
    # recall error from the GPU's final state against the oracle's, per pair, at
    # the state bar relative to the value's norm
    rg = _recall_errors(got["S_T"], x.keys, x.values)
    ro = _recall_errors(ref["S_T"], x.keys, x.values)
    vn = np.linalg.norm(x.values, axis=-1)
    assert np.all(np.abs(rg - ro) <= TOL["bf16"] * vn), float(np.max(np.abs(rg - ro) / vn))
    print("\nrecall n=%d chunk=%d: gpu mean %.4f max %.4f, oracle mean %.4f max %.4f"
          % (n_pairs, chunk, rg.mean(), rg.max(), ro.mean(), ro.max()))


@pytest.mark.parametrize("n_pairs", [32, 64])
def test_recall_exact_after_the_writes(n_pairs):
    """The first 2n tokens alone (orthonormal keys, u = k_hat, each pair twice):
    the gates are the keys and S k_i = v_i up to the rounding of the keys to
    bf16; the GPU's recall error matches the oracle's."""
    x = make_recall_stream(2, 2, 3 * n_pairs, 64, n_pairs, seed=65, dtype="bf16")
    w = x.slice_heads(slice(None), slice(None))
    T = 2 * n_pairs
    for n in "qkvu":
        setattr(w, n, np.ascontiguousarray(getattr(x, n)[:, :, :T]))
    ref = oracle_ref(w)
    got = run_gpu(w, TC, chunk=64)
    compare(got, ref, "bf16")
    rg = _recall_errors(got["S_T"], x.keys, x.values)
    ro = _recall_errors(ref["S_T"], x.keys, x.values)
    vn = np.linalg.norm(x.values, axis=-1)
    assert np.all(ro <= 2e-2 * vn)  # exact recall up to the bf16 rounding of the keys
    assert np.all(np.abs(rg - ro) <= TOL["bf16"] * vn), float(np.max(np.abs(rg - ro) / vn))


@pytest.mark.parametrize("B,H,T,chunk,per,launches", [
    (1, 16, 2048, 128, 1, 5),  # 256 jobs a pass (0.84 of a wave): one queue launch
    (1, 3, 6000, 0, 2, 5),     # S-chunks of two A-chunks, ragged tail: a state pass waits on two flags
    (1, 1, 16384, 0, 7, 5),    # S-chunks of seven A-chunks
    (1, 16, 2432, 128, 1, 6),  # 304 jobs a pass, one full wave each: two launches
])
def test_launch_form(B, H, T, chunk, per, launches):
    """The device entry runs the gates and the state pass as one queue launch
    where a pass's last wave would be part full, else as two launches (the
    launch count tells them apart: Grams, prefix, passes, chain, output
    pass); both forms against the oracle."""
    x = make_inputs(B, H, T, 64, "bf16", seed=83)
    C, CA = vla.vla_chunk_lengths(B, H, T, 64, vla.VLA_BF16, TC, chunk)
    assert C // CA == per and C % CA == 0
    got = run_gpu(x, TC, chunk=chunk)
    assert vla.vla_last_launch_count() == launches
    compare(got, oracle_ref(x), "bf16")


def test_bounded_wait_expiry_in_queue_launch():
    """Test hook: the gates jobs of the d = 64 queue launch leave their flags
    unset, so every state pass's bounded wait expires (1 ms), sets the device
    error word and skips its job; the launch still ends, and the next call is
    normal."""
    x = make_inputs(1, 16, 2048, 64, "bf16", seed=522)
    q, k, v, u = to_device(x)
    assert vla.vla_debug_inject(1, 1_000_000) == vla.VLA_OK
    try:
        vla.vla_forward(q, k, v, u, x.lambda0, kernel=TC, chunk=128)
        assert vla.vla_last_launch_count() == 5  # the queue form
        assert vla.vla_device_status() == vla.VLA_ERR_TIMEOUT
    finally:
        vla.vla_debug_inject(0)
    assert vla.vla_device_status() == vla.VLA_OK
    compare(run_gpu(x, TC, chunk=128), oracle_ref(x), "bf16")


def test_launch_form_queue_from_a_given_state():
    """The queue form from a given initial state: A0 is inverted first (one
    more launch); the first A-chunk starts from A0, later ones from the
    inverse of the prefix."""
    pre = make_inputs(1, 16, 300, 64, "bf16", seed=84)
    st = oracle_ref(pre)
    x = make_inputs(1, 16, 2048, 64, "bf16", seed=85)
    got = run_gpu(x, TC, S0=st["S_T"], A0=st["A_T"], n0=st["n_T"], chunk=128)
    assert vla.vla_last_launch_count() == 6
    compare(got, oracle_ref(x, S0=st["S_T"], A0=st["A_T"], n0=st["n_T"]), "bf16")
