"""Error metrics shared by the GPU parity tests (the benchmark spec's tolerances)."""
import numpy as np

OUT_MAX_REL_RMS = 1e-2      # max |err| <= 1e-2 * RMS(reference)
OUT_MEAN_REL = 2e-3         # sum |err| / sum |reference| <= 2e-3


def metrics(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    rms = float(np.sqrt((ref ** 2).mean()))
    return dict(max_err=float(err.max()), rms=rms, max_rel_rms=float(err.max() / rms),
                mean_rel=float(err.sum() / np.abs(ref).sum()))


def assert_close(got, ref, max_rel_rms=OUT_MAX_REL_RMS, mean_rel=OUT_MEAN_REL, what=""):
    m = metrics(got, ref)
    assert m["max_rel_rms"] <= max_rel_rms and m["mean_rel"] <= mean_rel, (what, m)
    return m


def bf16_ulp_distance(a_bf16_as_f64, b_bf16_as_f64):
    """Distance in bf16 steps between two arrays of bf16 values (as float64)."""
    a = np.asarray(a_bf16_as_f64, np.float32).view(np.uint32) >> 16
    b = np.asarray(b_bf16_as_f64, np.float32).view(np.uint32) >> 16
    # map sign-magnitude to a monotone integer line
    def mono(v):
        v = v.astype(np.int64)
        return np.where(v & 0x8000, -(v & 0x7FFF), v)
    return np.abs(mono(a) - mono(b))
