"""The deterministic test inputs of inferno.rs "IV.4: One command buffer per
token", section "The correctness ladder": a 64-bit LCG mapped to [-1, 1) in f32
and the Q8_0 fabricator that writes scale bytes 00 2c (f16 0.0625) and quants
(rng * 127) truncated to i8."""
import numpy as np

_MASK = (1 << 64) - 1


class P1Rng:
    def __init__(self, seed: int):
        self.state = seed & _MASK

    def f32(self) -> np.float32:
        self.state = (self.state * 6364136223846793005 + 1442695040888963407) & _MASK
        return np.float32(np.float32(self.state >> 33) / np.float32(1 << 31)) - np.float32(1.0)

    def vec(self, n: int) -> np.ndarray:
        return np.array([self.f32() for _ in range(n)], dtype=np.float32)


def random_q8_bytes(rows: int, cols: int, seed: int) -> np.ndarray:
    rng = P1Rng(seed)
    out = []
    for _ in range(rows * (cols // 32)):
        out += [0x00, 0x2C]
        for _ in range(32):
            v = np.float32(rng.f32() * np.float32(127.0))
            q = int(np.trunc(v))
            q = max(-128, min(127, q))
            out.append(q & 0xFF)
    return np.array(out, dtype=np.uint8).reshape(rows, cols // 32 * 34)
