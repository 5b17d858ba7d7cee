"""Small helpers shared by the tests (torch <-> numpy views; error metrics)."""
import numpy as np
import torch


def bits16(t: torch.Tensor) -> np.ndarray:
    """bf16 torch tensor -> numpy uint16 bit patterns (a view, no arithmetic)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy().view(np.uint8)


def bf16_values(t: torch.Tensor) -> np.ndarray:
    """bf16 torch tensor -> numpy float32 with the same values (torch does the widening)."""
    return t.detach().cpu().float().numpy()


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def cosine(a, b) -> float:
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    return float(a @ b / max(np.linalg.norm(a) * np.linalg.norm(b), 1e-30))


def oracle_args(inp):
    """Workload inputs (torch CPU tensors) -> the oracle's numpy argument tuple."""
    x = bits16(inp["x"])
    scores = inp["scores"].numpy()
    if inp["w1"].dtype == torch.bfloat16:
        w1, w2 = bits16(inp["w1"]), bits16(inp["w2"])
    else:
        w1, w2 = u8(inp["w1"]), u8(inp["w2"])
    s1 = None if inp["w1_scale"] is None else inp["w1_scale"].numpy()
    s2 = None if inp["w2_scale"] is None else inp["w2_scale"].numpy()
    return x, scores, w1, w2, s1, s2
