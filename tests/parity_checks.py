"""Shared tolerance checks of the GPU parity tests (not a test module).

Tolerances (GPU output widened to fp64, compared over the compared slice):
  O     max-abs <= 1e-2 beyond the output's own bf16 rounding (half an ulp of the
        exact value; above |O| = 4 that half ulp alone exceeds 1e-2), and
        normwise relative <= 5e-3
  LSE   max-abs <= 1e-3
  dQ/dK/dV  normwise relative <= 2e-2 each
"""
import numpy as np

O_ABS, O_REL, LSE_ABS, G_REL = 1e-2, 5e-3, 1e-3, 2e-2


def bf16_half_ulp(x):
    """Half the bf16 spacing at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -126)
    return np.ldexp(1.0, (np.floor(np.log2(ax)) - 8).astype(np.int64))


def relF(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def assert_o_close(got, ref):
    """O within the stated tolerance beyond bf16 rounding; returns the raw max-abs error
    (before the half-ulp allowance) so callers can report it."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    raw = np.abs(got - ref)
    excess = raw - bf16_half_ulp(ref)
    assert np.max(excess) <= O_ABS, float(np.max(excess))
    assert relF(got, ref) <= O_REL, relF(got, ref)
    return float(np.max(raw)) if raw.size else 0.0


def check_full(g, ref):
    """Every output of a GPU run (dict of tensors) against the full oracle (dict of fp64 arrays).
    Returns the raw O max-abs error."""
    out = g["out"].double().cpu().numpy()
    lse = g["lse"].double().cpu().numpy()
    raw = assert_o_close(out, ref["out"])
    assert np.max(np.abs(lse - ref["lse"])) <= LSE_ABS
    scale = max(float(np.linalg.norm(ref[key])) for key in ("dq", "dk", "dv") if key in g) if "dv" in g else 0.0
    for key in ("dq", "dk", "dv"):
        if key not in g:
            continue
        got = g[key].double().cpu().numpy()
        if np.linalg.norm(ref[key]) == 0.0:
            # exactly zero in the definition (window 1: every row attends only itself, so
            # dS = P (dP - Delta) = 0); the GPU result holds only the rounding of Delta,
            # bounded on the scale of the layer's other gradients
            assert np.linalg.norm(got) <= G_REL * scale, (key, float(np.linalg.norm(got)))
            continue
        assert relF(got, ref[key]) <= G_REL, (key, relF(got, ref[key]))
    return raw
