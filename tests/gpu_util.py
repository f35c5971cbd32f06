"""Small helpers shared by the GPU tests: numpy <-> device tensors (same bytes)."""
import numpy as np
import torch


def dev(a: np.ndarray) -> torch.Tensor:
    """Upload a numpy array to cuda:0 keeping its bytes (uint16 -> int16, uint8 -> uint8)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    elif a.dtype == np.uint32:
        a = a.view(np.int32)
    elif a.dtype == np.uint64:
        a = a.view(np.int64)
    return torch.from_numpy(a.copy()).to("cuda")


def host(t: torch.Tensor, dtype=None) -> np.ndarray:
    a = t.detach().cpu().numpy()
    if dtype is not None:
        a = a.view(dtype)
    return a


def bits_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    """Bitwise equality of two tensors of the same shape and dtype."""
    if a.shape != b.shape or a.dtype != b.dtype:
        return False
    ai = a.contiguous().view(torch.int32) if a.element_size() == 4 else a.contiguous().view(torch.int16)
    bi = b.contiguous().view(torch.int32) if b.element_size() == 4 else b.contiguous().view(torch.int16)
    return bool(torch.equal(ai, bi))


def rel_err_rows(got: np.ndarray, ref: np.ndarray) -> float:
    """max over rows of max|got - ref| / max|ref| of that row (rows = last axis vectors)."""
    got = got.reshape(-1, got.shape[-1]).astype(np.float64)
    ref = ref.reshape(-1, ref.shape[-1]).astype(np.float64)
    scale = np.maximum(np.abs(ref).max(axis=1), 1e-30)
    return float((np.abs(got - ref).max(axis=1) / scale).max())


TOL = 2e-3  # max abs error relative to the output row's max-abs (fp32-accumulated 16-bit math)


def bf16_round(x) -> np.ndarray:
    """float64 values rounded to bfloat16 (8 significant bits, ties to even), as float64."""
    x = np.asarray(x, np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0), e - 8)


def bf16_rounding_report(got_bits: np.ndarray, ref: np.ndarray, slack) -> str:
    """The elements bf16_rounding_ok rejects, for a failure message."""
    got = bits_to_f64(got_bits).reshape(-1)
    ref = np.asarray(ref, np.float64).reshape(-1)
    slack = np.broadcast_to(np.asarray(slack, np.float64), ref.shape).reshape(-1)
    exp = bf16_round(ref)
    lo, hi = bf16_round(ref - slack), bf16_round(ref + slack)
    bad = np.nonzero((got < lo) | (got > hi) | np.isnan(got))[0]
    return "; ".join(f"[{i}] got {got[i]!r} ref {ref[i]!r} rounded {exp[i]!r} slack {slack[i]:.3g}" for i in bad[:6])


def bf16_rounding_ok(got_bits: np.ndarray, ref: np.ndarray, slack) -> bool:
    """A bf16 output that rounds a quantity whose exact value is ``ref``, computed
    on the device within ``slack`` (absolute, per element) of it.  Rounding to
    nearest is monotone, so every element lies between ref - slack and
    ref + slack, each rounded to bf16: ref rounded itself when the slack stays
    inside one rounding interval, either neighbour near a midpoint, and a run of
    bf16 values where the slack spans several (a cancellation, whose absolute
    error is set by the operands, not by the result)."""
    got = bits_to_f64(got_bits)
    ref = np.asarray(ref, np.float64)
    slack = np.broadcast_to(np.asarray(slack, np.float64), ref.shape)
    exp = bf16_round(ref)
    bad = got != exp
    if not bad.any():
        return True
    lo, hi = bf16_round(ref[bad] - slack[bad]), bf16_round(ref[bad] + slack[bad])
    g = got[bad]
    return bool(np.all((g >= lo) & (g <= hi)))


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits).view(np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
