"""Helpers shared by the GPU parity tests (no method arithmetic here)."""
import numpy as np

# fp16 outputs: |got - ref| <= ATOL + RTOL * |ref| elementwise, ref = oracle (fp64, one fp16 rounding)
ATOL = 1e-2
RTOL = 2e-3


def to_dev(a, torch):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).cuda()


def to_host(t):
    return t.detach().cpu().numpy()


def assert_close(got, ref, atol=ATOL, rtol=RTOL, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"got {got[i]} ref {ref[i]} (err {err[i]:.3g}, bound {bound[i]:.3g})")


def max_rel(got, ref, floor=1e-2):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    m = np.abs(ref) > floor
    return float(np.max(np.abs(got[m] - ref[m]) / np.abs(ref[m]))) if m.any() else 0.0


def assert_close_composite(got, ref, atol=ATOL, rtol=RTOL, what=""):
    """Bound for outputs composed of several fp16-rounded operations (a whole
    decoder layer): a 1-ulp flip in an intermediate rounding moves the output
    by an amount that scales with the output's RMS, not with each element, so
    the relative part of the bound uses max(|ref|, rms(ref))."""
    ref64 = np.asarray(ref, dtype=np.float64)
    scale = np.maximum(np.abs(ref64), np.sqrt(np.mean(ref64 ** 2)))
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref64)
    bound = atol + rtol * scale
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"got {got[i]} ref {ref64[i]} (err {err[i]:.3g}, bound {bound[i]:.3g})")
