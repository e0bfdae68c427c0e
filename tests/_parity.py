"""Shared helpers of the parity tests: bf16 views for the oracle, the
tolerance of the layer's bf16 outputs, and a lazily-copied weight view so
the oracle can read only the experts a sampled token touches."""
import numpy as np
import torch

from lora_mixture_experts_gb300.inputs import bf16_bits

# bf16 outputs with fp32 accumulation: relative Frobenius error <= 1e-2 and
# max-abs error <= 3e-2 x RMS of the oracle output.
REL_FRO_TOL = 1e-2
MAX_ABS_RMS_TOL = 3e-2


class LazyBf16:
    """Indexable view of a (device) bf16 tensor that copies only the indexed
    slice to the host, as bf16 bit patterns."""

    def __init__(self, t: torch.Tensor):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, idx):
        return bf16_bits(self.t[idx])


def np_inputs(d, lazy=False):
    out = {}
    for k, v in d.items():
        if v.dtype == torch.bfloat16:
            out[k] = LazyBf16(v) if (lazy and k != "x") else bf16_bits(v)
        else:
            out[k] = v.cpu().numpy()
    return out


def compare(gpu_out: torch.Tensor, ref: np.ndarray, what=""):
    """Returns (ok, message) for the layer's tolerance."""
    g = gpu_out.float().cpu().numpy().astype(np.float64)
    diff = g - ref
    ref_norm = np.linalg.norm(ref)
    rel = np.linalg.norm(diff) / max(ref_norm, 1e-30)
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    maxabs = np.abs(diff).max() if ref.size else 0.0
    ok = bool(np.all(np.isfinite(g)) and rel <= REL_FRO_TOL and maxabs <= MAX_ABS_RMS_TOL * max(rms, 1e-30))
    msg = f"{what}: rel_fro={rel:.3e} max_abs={maxabs:.3e} rms={rms:.3e}"
    if not ok and ref.size:
        i = np.unravel_index(np.argmax(np.abs(diff)), diff.shape)
        msg += f" worst at {tuple(int(v) for v in i)}: gpu={g[i]:.5f} ref={ref[i]:.5f}"
    return ok, msg
