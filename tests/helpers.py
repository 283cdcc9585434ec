"""Small test helpers: golden-file parsing and dtype views (no method arithmetic)."""
import os

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_golden(name):
    """Parse tests/golden/<name> lines 'key: v v v' into {key: [int, ...]}."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, vals = line.split(":", 1)
            out[key.strip()] = [int(v) for v in vals.split()]
    return out


def bf16_bits(values):
    """uint16 bit patterns of `values` rounded to bf16 by torch."""
    t = torch.as_tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_values(bits):
    """float64 values of uint16 bf16 bit patterns, converted by torch."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.double().numpy()


def bf16_half_ulp(ref):
    """Half a bf16 ulp at |ref|: the largest error of rounding the exact value
    to the bf16 output (bf16 carries 8 significant bits)."""
    ref = np.abs(np.asarray(ref, dtype=np.float64))
    _, e = np.frexp(ref)           # ref = m * 2**e, 0.5 <= m < 1
    # below 2^-126 bf16 is subnormal: its spacing stays 2^-133
    h = np.maximum(np.ldexp(1.0, e - 9), 2.0 ** -134)
    return np.where(ref > 0, h, 0.0)


def parity_violations(got, ref, ref_abs, tol, bf16_out):
    """Boolean mask of outputs outside |got - ref| <= tol * ref_abs (+ the
    half-ulp rounding of a bf16 output).  The accumulation tolerance bounds
    the value before it is stored; storing it as bf16 adds at most half an
    ulp, which alone can exceed tol * ref_abs when |ref| is close to ref_abs
    (short K)."""
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    bound = tol * ref_abs + (bf16_half_ulp(ref) if bf16_out else 0.0)
    return err > bound
