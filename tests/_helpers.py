"""Small host helpers shared by the GPU parity tests (no method arithmetic)."""
import numpy as np


def cuda_ready():
    import torch
    return torch.cuda.is_available()


def dev_bf16(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t) -> np.ndarray:
    return t.detach().cpu().numpy()


def unpack(q: np.ndarray) -> np.ndarray:
    out = np.empty((q.shape[0], q.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = q & 0xF
    out[:, 1::2] = q >> 4
    return out


def mma_scale_index(rows: int, scols: int) -> np.ndarray:
    """Byte offset of each scale (r, c) in the 128x4-tile MMA layout, as an int64 [rows, scols] array."""
    r = np.arange(rows, dtype=np.int64)[:, None]
    c = np.arange(scols, dtype=np.int64)[None, :]
    s4 = (scols + 3) // 4
    return ((r // 128) * s4 + c // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (c % 4)


def from_mma_layout(buf: np.ndarray, rows: int, scols: int) -> np.ndarray:
    return buf[mma_scale_index(rows, scols)]


def to_mma_layout(s: np.ndarray) -> np.ndarray:
    rows, scols = s.shape
    out = np.zeros(((rows + 127) // 128) * ((scols + 3) // 4) * 512, dtype=np.uint8)
    out[mma_scale_index(rows, scols)] = s
    return out


def rel_frobenius(y, ref) -> float:
    """||y - ref||_F / ||ref||_F in float64 (the GEMM parity measure)."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(y - ref) / (den if den > 0 else 1.0))
