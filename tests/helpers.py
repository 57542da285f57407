"""Shared test helpers: host-side packing of q8 records and running one layer
through the CUDA library.  The oracle never sees a value produced by the
CUDA path; inputs flow from the generator (and the oracle) to the GPU only."""
import numpy as np

TOL_REL, TOL_ABS = 1e-3, 1e-5   # y: max|err| <= 1e-3 * max|y_ref| + 1e-5


def act_block(n):
    return 256 if n % 256 == 0 else 32


def q8_row_bytes(n):
    B = act_block(n)
    a = (4 * (n // B) + 15) & ~15
    return (a + n + 2 * (n // 16) + 15) & ~15


def pack_q8_records(d, q, bs):
    """oracle (d [T, n/B], q [T, n], bsum [T, n/16]) -> q8 record bytes [T * row_bytes]"""
    d, q, bs = np.atleast_2d(d), np.atleast_2d(q), np.atleast_2d(bs)
    T, n = q.shape
    B = n // d.shape[1]
    rb = q8_row_bytes(n)
    a = (4 * (n // B) + 15) & ~15
    out = np.zeros((T, rb), np.uint8)
    out[:, :4 * (n // B)] = d.astype(np.float32).view(np.uint8).reshape(T, -1)
    out[:, a:a + n] = q.astype(np.int8).view(np.uint8)
    out[:, a + n:a + n + 2 * (n // 16)] = bs.astype(np.int16).view(np.uint8).reshape(T, -1)
    return out.reshape(-1)


def unpack_q8_records(buf, T, n):
    B = act_block(n)
    rb = q8_row_bytes(n)
    a = (4 * (n // B) + 15) & ~15
    r = np.asarray(buf)[:T * rb].reshape(T, rb)
    d = r[:, :4 * (n // B)].copy().view(np.float32)
    q = r[:, a:a + n].copy().view(np.int8)
    bs = r[:, a + n:a + n + 2 * (n // 16)].copy().view(np.int16)
    return d, q, bs


def y_tol(y_ref):
    return TOL_REL * float(np.max(np.abs(y_ref))) + TOL_ABS


def assert_y_close(y_gpu, y_ref, what=""):
    err = float(np.max(np.abs(np.asarray(y_gpu, np.float64) - y_ref)))
    tol = y_tol(y_ref)
    assert err <= tol, f"{what}: max|err| {err:.3e} > tol {tol:.3e} (max|y| {np.max(np.abs(y_ref)):.3e})"
    return err
