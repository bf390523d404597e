"""Comparison helpers for the CUDA-vs-oracle parity tests.

Tolerances are the ones the workloads fix:
  fp32 storage:       relative L2 <= 1e-5 and max-abs <= 1e-4
  fp16/bf16 storage:  relative L2 <= 2e-2 and cosine >= 0.9999
plus an element-wise bound derived from the arithmetic, so that a localised
error (one wrong channel, one wrong tap at an edge) cannot hide inside a
norm: a stored fp16/bf16 result is the fp32 accumulation rounded once, so it
lies within one unit in the last place of the fp64 value, i.e.
|gpu - ref| <= 2^-(p-1) |ref| + 1e-3 * max|ref| (p = 8 for bf16, 11 for fp16;
the absolute term covers fp32 accumulation error on cancelling sums).
"""
import numpy as np
import torch

REL_L2_F32, MAX_ABS_F32 = 1e-5, 1e-4
REL_L2_LOW, COS_LOW = 2e-2, 0.9999
SIG_BITS = {torch.bfloat16: 8, torch.float16: 11}


def to64(t) -> np.ndarray:
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu", torch.float64).numpy()


def metrics(got, ref):
    g, r = to64(got).ravel(), to64(ref).ravel()
    d = g - r
    nr = np.linalg.norm(r)
    rel = np.linalg.norm(d) / nr if nr > 0 else np.linalg.norm(d)
    cos = float(g @ r / (np.linalg.norm(g) * nr)) if nr > 0 and np.linalg.norm(g) > 0 else 1.0
    return {"rel_l2": float(rel), "max_abs": float(np.abs(d).max(initial=0.0)), "cos": cos}


def assert_parity(got, ref, dtype, what=""):
    """`got` (GPU output, any torch dtype) against the fp64 oracle `ref`."""
    g, r = to64(got), to64(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite GPU output"
    m = metrics(g, r)
    if dtype == torch.float32:
        assert m["rel_l2"] <= REL_L2_F32 and m["max_abs"] <= MAX_ABS_F32, (what, m)
    else:
        assert m["rel_l2"] <= REL_L2_LOW and m["cos"] >= COS_LOW, (what, m)
        p = SIG_BITS[dtype]
        bound = 2.0 ** (1 - p) * np.abs(r) + 1e-3 * np.abs(r).max(initial=0.0)
        bad = np.abs(g - r) > bound
        assert not bad.any(), (what, m, int(bad.sum()), np.argwhere(bad)[:5].tolist())
    return m


def assert_bitexact(got, ref, what=""):
    g, r = to64(got), to64(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    bad = g != r
    assert not bad.any(), (what, int(bad.sum()), np.argwhere(bad)[:5].tolist())


# A byte of the flow-out stage is trunc(v * 255) of a binary32 value v in
# [0, 1].  Kernel and oracle compute v in the same binary32 operation order
# except for the mask's exp (CUDA's expf, within 2 ulp; the C library's
# double exp rounded to float, within 1 ulp), which moves the sigmoid m by at
# most ~3 ulp (< 2e-7) and the blended v by < 1e-6; times 255 that is < 3e-4.
# So a byte may differ by one only where the oracle's v * 255 lies within
# BYTE_WINDOW of an integer; everywhere else the bytes must be equal.
BYTE_WINDOW = 5e-4


def assert_bytes_boundary(got, ref, pre, what=""):
    """`got`, `ref`: [H, W, 4] uint8 (R, G, B, A); `pre`: the oracle's clamped
    R, G, B values [3, H, W] before the byte scale.  Returns the number of
    channel values that differ by one at a byte boundary (all others equal)."""
    g = got.detach().cpu().numpy().astype(np.int32) if isinstance(got, torch.Tensor) \
        else np.asarray(got, np.int32)
    r = np.asarray(ref, np.int32)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert (g[..., 3] == r[..., 3]).all(), f"{what}: alpha differs"
    d = g[..., :3] - r[..., :3]
    scaled = np.moveaxis(np.asarray(pre, np.float64), 0, -1) * 255.0
    near = np.abs(scaled - np.rint(scaled)) <= BYTE_WINDOW
    bad = (d != 0) & ~((np.abs(d) == 1) & near)
    assert not bad.any(), (what, int(bad.sum()), np.argwhere(bad)[:5].tolist())
    n1 = int((d != 0).sum())
    print(f"{what}: {n1} of {d.size} channel bytes differ by 1 at a byte boundary "
          f"({int(near.sum())} values within {BYTE_WINDOW} of one)")
    return n1


# Canary guards: the compute-sanitizer's out-of-bounds check is closed on this
# pool, so every output (and workspace) of the op tests lives inside a byte
# buffer whose GUARD bytes before and after it hold a canary pattern; a store
# past either end (a ragged tile tail written too far) changes them.  The
# interior starts as the same pattern (0xFF bytes are NaN in fp32, fp16 and
# bf16), so an element the op forgot to write stays NaN and fails the parity
# check's finiteness test.
GUARD = 4096
CANARY = 0xFF


class Guarded:
    """A device tensor of `shape`/`dtype` with canary bytes on both sides."""

    def __init__(self, shape, dtype, device="cuda"):
        shape = tuple(int(s) for s in shape)
        es = torch.empty((), dtype=dtype).element_size()
        self.nbytes = int(np.prod(shape, dtype=np.int64)) * es
        self.raw = torch.full((GUARD + self.nbytes + GUARD,), CANARY, dtype=torch.uint8,
                              device=device)
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(shape)

    def check(self, what=""):
        torch.cuda.synchronize()
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.nbytes:]
        bad_h = int((head != CANARY).sum())
        bad_t = int((tail != CANARY).sum())
        assert bad_h == 0 and bad_t == 0, f"{what}: {bad_h} bytes before and {bad_t} after " \
                                          f"the buffer were overwritten"


def guarded_bytes(nbytes, device="cuda"):
    """A uint8 workspace of nbytes (None for 0) with canaries on both sides."""
    return Guarded((nbytes,), torch.uint8, device) if nbytes else None
