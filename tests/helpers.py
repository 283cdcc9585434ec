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
