"""Helpers shared by the GPU tests: host<->device copies of bit patterns and the tolerances.

Tolerances (stated once, used everywhere):
  - bf16 outputs vs the oracle: max|err| <= 2e-2 * RMS(reference);
  - fp32 GDN state vs the oracle (same bf16 inputs on both sides):
    max_i |d_i| / max(|ref_i|, RMS(ref)) <= 1e-4;
  - fp32 logits of the whole block vs the oracle's sequential decode:
    every row's RMS(err) <= 3 * the largest row RMS(spread) and max|err| <=
    3 * max|spread|, where spread is the oracle's own single-precision
    evaluation minus its double one on the same inputs (the same rows,
    extended on the tiny blocks to 64 positions of the same sequence, whose
    few rounding flips per row otherwise leave rows without any).  A block output has passed through ~8
    bf16 storage points per layer; a value that lands within the fp32
    accumulation error of a bf16 rounding boundary rounds the other way in
    any fp32 evaluation, and those 1-ulp differences propagate: the spread
    measures how far a faithful fp32 evaluation lands from the exact one, and
    the factor 3 leaves room for the device's different (equally valid)
    accumulation order.  Argmax ids equal the lowest-index maximum of the
    GPU's own logits row (exactly), and the oracle's argmax wherever the
    oracle's top-1/top-2 margin exceeds twice the max bound (no pair of
    logits within the bound can swap there); each such check must find a
    decisive row;
  - one layer of the stack, teacher forced (the oracle's layer fed the GPU's
    own bf16 residual input x and the same layer state): the layer is
    x -> mid = bf16(x + y1) -> out = bf16(mid + y2) with y1 the mixer's and y2
    the MLP's bf16 output.  If each of y1, y2 carries at most the per-output
    error 2e-2 * RMS and each residual sum rounds the other way at most once
    (a flip costs the bf16 spacing at that element), element i satisfies
    |err_i| <= 2e-2 * (RMS(y1) + RMS(y2)) + spacing(mid_i) + spacing(out_i)
    (y1, y2, mid, out from the double oracle).  The MLP is three storage
    points deep, and on the 5120-wide stack its 17408 bf16 SwiGLU values, each
    of which may round the other way, move a faithful single-precision
    evaluation of y2 by up to 2.3% of RMS(y2) at the worst of 10240 elements,
    past that bound; so element i may also deviate by up to 3 * max|spread|,
    the spread being the single-precision oracle's layer output minus the
    double one on the same inputs (as for the logits).  RMS(err) <=
    max(2e-2 * RMS(out - x), 3 * RMS(spread)).  (The bare 2e-2 * RMS(out) per
    element rejects the single-precision evaluation there too: one flip at an
    element of magnitude 16..32 costs 0.125.)
  - GPU vs GPU comparisons: 0 differing bits.
"""
import numpy as np
import torch

BF16_REL = 2e-2
STATE_REL = 1e-4


def dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda()
    return torch.from_numpy(a).cuda()


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def f64(u16: np.ndarray) -> np.ndarray:
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rms(x) -> float:
    x = np.asarray(x, dtype=np.float64)
    return float(np.sqrt(np.mean(x * x)))


def assert_bf16_close(got_u16, ref, rel=BF16_REL, what=""):
    """got: bf16 bits; ref: bf16 bits (uint16) or float values."""
    g = f64(got_u16)
    r = f64(ref) if np.asarray(ref).dtype == np.uint16 else np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    err = float(np.max(np.abs(g - r))) if g.size else 0.0
    bound = rel * rms(r)
    assert err <= bound, f"{what}: max|err| {err:.3e} > {rel} * RMS = {bound:.3e}"
    return err / max(rms(r), 1e-300)


def assert_f32_close(got, ref, rel=BF16_REL, what=""):
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    err = float(np.max(np.abs(g - r)))
    bound = rel * rms(r)
    assert err <= bound, f"{what}: max|err| {err:.3e} > {rel} * RMS = {bound:.3e}"


SPREAD_FACTOR = 3.0


def assert_block_close(got, ref, spread, what=""):
    """got, ref: fp32/fp64 logits [n, V]; spread: f32-oracle minus f64-oracle logits on the same
    inputs (at least the compared rows).  Returns the max-error bound."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    sp = np.asarray(spread, dtype=np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    row_rms = lambda x: np.sqrt(np.mean(x.reshape(x.shape[0], -1) ** 2, axis=1))
    rms_bound, max_bound = SPREAD_FACTOR * float(row_rms(sp).max()), SPREAD_FACTOR * float(np.max(np.abs(sp)))
    assert rms_bound > 0 and max_bound > 0, f"{what}: degenerate spread"
    e = np.abs(g - r).reshape(g.shape[0] if g.ndim > 1 else 1, -1)
    worst = float(row_rms(e).max())
    assert worst <= rms_bound, f"{what}: row RMS err {worst:.3e} > {SPREAD_FACTOR} * max row RMS(spread) = {rms_bound:.3e}"
    assert e.max() <= max_bound, f"{what}: max err {e.max():.3e} > {SPREAD_FACTOR} * max|spread| = {max_bound:.3e}"
    return max_bound


def assert_argmax(ids, got, ref, max_bound, min_decisive=1):
    """ids: GPU argmax [n]; got: the GPU logits [n, V] they came from; ref: oracle logits [n, V].
    Every id is the lowest-index maximum of its GPU row; where the oracle's top-1/top-2 margin
    exceeds 2 * max_bound it is also the oracle's argmax.  Returns the number of such rows, which
    must be at least min_decisive."""
    ids = np.asarray(ids).reshape(-1)
    got = np.asarray(got)
    assert np.array_equal(ids, np.argmax(got, axis=1)), "argmax is not the lowest-index maximum of the logits"
    decisive = 0
    for i, r in zip(ids, np.asarray(ref, dtype=np.float64)):
        top2 = np.partition(r, -2)[-2:]
        if top2[1] - top2[0] > 2 * max_bound:
            assert int(i) == int(np.argmax(r)), f"argmax {int(i)} != oracle {int(np.argmax(r))} (margin {top2[1] - top2[0]:.3f})"
            decisive += 1
    assert decisive >= min_decisive, f"{decisive} decisive rows (margin > {2 * max_bound:.3e}), {min_decisive} needed"
    return decisive


def bf16_spacing(v) -> np.ndarray:
    """The gap from |v| to the next bf16 value above it, 2^(floor(log2 |v|) - 7); 0 at 0."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, e = np.frexp(a)
    return np.where(a > 0, np.ldexp(1.0, e - 8), 0.0)


def layer_bound(x_in, mid, out, rel=BF16_REL):
    """The per-element bound and the RMS bound of a teacher-forced layer output from the
    per-output error and the residual roundings alone (bf16 bits of the residual input, the
    oracle's mid residual and its output; see the module docstring)."""
    x, m, o = f64(x_in), f64(mid), f64(out)
    per = rel * (rms(m - x) + rms(o - m)) + bf16_spacing(m) + bf16_spacing(o)
    return per, rel * rms(o - x)


def assert_layer_close(got_u16, x_in, mid, out, out32, rel=BF16_REL, what=""):
    """got: the GPU's layer output (bf16 bits [n, H]); x_in its residual input; mid, out: the
    double oracle's layer run on x_in, out32 the single-precision oracle's.  Returns the largest
    err / per-element bound."""
    g = f64(got_u16)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    per, rms_bound = layer_bound(x_in, mid, out, rel)
    spread = f64(out32) - f64(out)
    per = np.maximum(per, SPREAD_FACTOR * float(np.max(np.abs(spread))))
    rms_bound = max(rms_bound, SPREAD_FACTOR * rms(spread))
    e = np.abs(g - f64(out))
    worst = float(np.max(e / per))
    i = np.unravel_index(int(np.argmax(e / per)), e.shape)
    assert worst <= 1.0, f"{what}: err {e[i]:.3e} at {i} > bound {per[i]:.3e}"
    assert rms(e) <= rms_bound, f"{what}: RMS err {rms(e):.3e} > {rel} * RMS(out - x) = {rms_bound:.3e}"
    return worst


def assert_state_close(got, ref, rel=STATE_REL, what="state"):
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    floor = np.maximum(np.abs(r), rms(r))
    worst = float(np.max(np.abs(g - r) / floor))
    assert worst <= rel, f"{what}: max rel err {worst:.3e} > {rel}"
    return worst


def same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    if a.shape != b.shape:
        return False
    if a.dtype in (torch.float32,):
        return torch.equal(a.view(torch.int32), b.view(torch.int32))
    if a.element_size() == 2:
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    return torch.equal(a, b)
