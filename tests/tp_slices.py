"""Numpy statement of a tensor-parallel weight slice along I (part p of
`parts`): rows [p Is, (p+1) Is) of gate and up, the same columns of down,
with the Int4 codes (two per byte) and group-of-32 scales cut at the same
places.  The GPU tests hold moe_tp_slice_weights to it bit for bit, and the
gloo test runs the oracle on it."""
from __future__ import annotations

import numpy as np


def slice_stack(stack: dict, part: int, parts: int) -> dict:
    I = stack["gate"].shape[1]
    Is = I // parts
    r = slice(part * Is, (part + 1) * Is)
    out = {"gate": stack["gate"][:, r], "up": stack["up"][:, r]}
    if "gate_scale" in stack:  # Int4: codes [n][H][I/2], scales [n][H][I/32]
        out["down"] = stack["down"][:, :, part * Is // 2:(part + 1) * Is // 2]
        out["gate_scale"] = stack["gate_scale"][:, r]
        out["up_scale"] = stack["up_scale"][:, r]
        out["down_scale"] = stack["down_scale"][:, :, part * Is // 32:(part + 1) * Is // 32]
    else:
        out["down"] = stack["down"][:, :, r]
    return {k: np.ascontiguousarray(v) for k, v in out.items()}
