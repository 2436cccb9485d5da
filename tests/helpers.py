"""Shared test helpers: tolerance checks and device plumbing."""
import numpy as np

# Tolerance for fp32-accumulated products against the fp64 oracle: 1e-3
# max-rel, read as (a) normwise  max|y - yref| / max|yref|  and (b)
# componentwise  max|y - yref| / sum_k |w x|  (the two readings of "max-rel"
# that stay meaningful where yref is near zero).
TOL = 1e-3


def rel_errors(y, yref, absprod):
    y = np.asarray(y, dtype=np.float64)
    yref = np.asarray(yref, dtype=np.float64)
    d = np.abs(y - yref)
    normwise = d.max() / max(np.abs(yref).max(), 1e-300)
    compwise = (d / np.maximum(np.asarray(absprod, dtype=np.float64), 1e-300)).max()
    return float(normwise), float(compwise)


def assert_close(y, yref, absprod, tol=TOL):
    nw, cw = rel_errors(y, yref, absprod)
    assert nw <= tol and cw <= tol, f"normwise {nw:.3e}, componentwise {cw:.3e} > {tol}"
    return nw, cw


def cuda_tensors(torch, *arrays, device="cuda"):
    return [torch.from_numpy(np.ascontiguousarray(a)).to(device) for a in arrays]
