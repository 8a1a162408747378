"""Small helpers shared by the tests (marshalling between numpy bit patterns and
torch tensors, error norms). No arithmetic of the method lives here."""
import numpy as np

try:
    import torch
except Exception:  # pragma: no cover
    torch = None


def bf16_dev(bits, dev="cuda"):
    """uint16 bf16 bit patterns -> a bf16 CUDA tensor."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def f32_dev(a, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)


def host(t):
    """A CUDA tensor -> numpy (bf16 -> float64 values, uint8 stays uint8)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.float().numpy().astype(np.float64)
    if t.dtype == torch.uint8:
        return t.numpy()
    return t.numpy()


def rel_fro(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def f32_bits(x):
    return np.asarray(x, np.float32).view(np.uint32)
