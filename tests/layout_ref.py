"""A numpy statement of the repacked Q4_0 layout documented in include/gq.h,
written from that description for the GPU tests (host logic, not the oracle)."""
import numpy as np


def repack_ref(q4: np.ndarray) -> np.ndarray:
    """Canonical Q4_0 bytes [N, nb, 18] -> repacked bytes [N16 * NT * 1152]."""
    N, nb = q4.shape[0], q4.shape[1]
    N16, NT = -(-N // 16), -(-nb // 4)
    P = np.zeros((N16 * 16, NT * 4, 18), np.uint8)
    P[..., 2:] = 0x88
    P[:N, :nb] = q4
    T = P.reshape(N16, 16, NT, 4, 18).transpose(0, 2, 3, 1, 4)   # [g, t, j, r, 18]
    out = np.empty((N16, NT, 1152), np.uint8)
    out[:, :, :1024] = T[..., 2:].reshape(N16, NT, 1024)
    out[:, :, 1024:] = T[..., :2].transpose(0, 1, 3, 2, 4).reshape(N16, NT, 128)   # [r, j, 2]
    return out.reshape(-1)


def repack_loops(q4: np.ndarray) -> np.ndarray:
    """The same layout, byte by byte, in the words of the header (slow; small sizes)."""
    N, nb = q4.shape[0], q4.shape[1]
    N16, NT = -(-N // 16), -(-nb // 4)
    out = np.zeros(N16 * NT * 1152, np.uint8)
    for g in range(N16):
        for t in range(NT):
            base = (g * NT + t) * 1152
            for j in range(4):
                for r in range(16):
                    n, b = 16 * g + r, 4 * t + j
                    real = n < N and b < nb
                    for i in range(16):
                        out[base + (j * 16 + r) * 16 + i] = q4[n, b, 2 + i] if real else 0x88
                    for i in range(2):
                        out[base + 1024 + (r * 4 + j) * 2 + i] = q4[n, b, i] if real else 0
    return out


def repack_f16_ref(w16: np.ndarray) -> np.ndarray:
    """F16 bits [N, K] (uint16) -> the 16 x 32 tile layout of gq_repack_f16, as bytes."""
    N, K = w16.shape
    N16, NT = -(-N // 16), K // 32
    P = np.zeros((N16 * 16, K), np.uint16)
    P[:N] = w16
    T = P.reshape(N16, 16, NT, 32).transpose(0, 2, 1, 3)        # [g, t, r, c]
    return np.ascontiguousarray(T).reshape(-1).view(np.uint8)


def repack_f16_loops(w16: np.ndarray) -> np.ndarray:
    """The same layout element by element, in the words of the header (small sizes)."""
    N, K = w16.shape
    N16, NT = -(-N // 16), K // 32
    out = np.zeros(N16 * NT * 512, np.uint16)
    for g in range(N16):
        for t in range(NT):
            for r in range(16):
                for c in range(32):
                    n = 16 * g + r
                    out[((g * NT + t) * 1024 + r * 64 + 2 * c) // 2] = w16[n, 32 * t + c] if n < N else 0
    return out.view(np.uint8)


def repack_q8_0_ref(q8: np.ndarray) -> np.ndarray:
    """Q8_0 blocks [N, nb, 34] -> the tile layout of gq_repack_q8_0, as bytes."""
    N, nb = q8.shape[0], q8.shape[1]
    N16, NT = -(-N // 16), -(-nb // 4)
    P = np.zeros((N16 * 16, NT * 4, 34), np.uint8)
    P[:N, :nb] = q8
    T = P.reshape(N16, 16, NT, 4, 34).transpose(0, 2, 3, 1, 4)   # [g, t, j, r, 34]
    out = np.empty((N16, NT, 2176), np.uint8)
    out[:, :, :2048] = T[..., 2:].reshape(N16, NT, 2048)
    out[:, :, 2048:] = T[..., :2].transpose(0, 1, 3, 2, 4).reshape(N16, NT, 128)   # [r, j, 2]
    return out.reshape(-1)


def repack_q8_0_loops(q8: np.ndarray) -> np.ndarray:
    """The same layout, byte by byte, in the words of the header (small sizes)."""
    N, nb = q8.shape[0], q8.shape[1]
    N16, NT = -(-N // 16), -(-nb // 4)
    out = np.zeros(N16 * NT * 2176, np.uint8)
    for g in range(N16):
        for t in range(NT):
            base = (g * NT + t) * 2176
            for j in range(4):
                for r in range(16):
                    n, b = 16 * g + r, 4 * t + j
                    if n < N and b < nb:
                        out[base + (j * 16 + r) * 32: base + (j * 16 + r) * 32 + 32] = q8[n, b, 2:]
                        out[base + 2048 + (r * 4 + j) * 2: base + 2048 + (r * 4 + j) * 2 + 2] = q8[n, b, :2]
    return out


def _q5_high_word(qh: int) -> int:
    """The fifth bits of one block as gq_repack_q5_0 stores them (bit 8b + 7 - s = the fifth
    bit of element b of group s; groups 0..3 = elements 4s.., groups 4..7 = 16 + 4(s-4)..)."""
    h = 0
    for s in range(8):
        for b in range(4):
            e = 4 * s + b if s < 4 else 16 + 4 * (s - 4) + b
            h |= ((qh >> e) & 1) << (8 * b + 7 - s)
    return h


def repack_q5_0_ref(q5: np.ndarray) -> np.ndarray:
    """Q5_0 blocks [N, nb, 22] -> the tile layout of gq_repack_q5_0, as bytes (element by
    element from the header's description; small sizes)."""
    N, nb = q5.shape[0], q5.shape[1]
    N16, NT = -(-N // 16), -(-nb // 4)
    out = np.zeros(N16 * NT * 1408, np.uint8)
    pad_high = np.frombuffer(_q5_high_word(0xFFFFFFFF).to_bytes(4, "little"), np.uint8)
    for g in range(N16):
        for t in range(NT):
            base = (g * NT + t) * 1408
            for j in range(4):
                for r in range(16):
                    n, b = 16 * g + r, 4 * t + j
                    o_nib, o_hi, o_sc = base + (j * 16 + r) * 16, base + 1024 + (j * 16 + r) * 4, base + 1280 + (r * 4 + j) * 2
                    if n < N and b < nb:
                        out[o_nib:o_nib + 16] = q5[n, b, 6:22]
                        qh = int.from_bytes(bytes(q5[n, b, 2:6]), "little")
                        out[o_hi:o_hi + 4] = np.frombuffer(_q5_high_word(qh).to_bytes(4, "little"), np.uint8)
                        out[o_sc:o_sc + 2] = q5[n, b, 0:2]
                    else:
                        out[o_hi:o_hi + 4] = pad_high          # code 16: nibble 0, fifth bit 1; scale 0
    return out


def repack_q4_1_ref(q41: np.ndarray) -> np.ndarray:
    """Q4_1 blocks [N, nb, 20] -> the tile layout of gq_repack_q4_1, as bytes."""
    N, nb = q41.shape[0], q41.shape[1]
    N16, NT = -(-N // 16), -(-nb // 4)
    P = np.zeros((N16 * 16, NT * 4, 20), np.uint8)
    P[:N, :nb] = q41
    T = P.reshape(N16, 16, NT, 4, 20).transpose(0, 2, 3, 1, 4)   # [g, t, j, r, 20]
    out = np.empty((N16, NT, 1280), np.uint8)
    out[:, :, :1024] = T[..., 4:].reshape(N16, NT, 1024)
    out[:, :, 1024:1152] = T[..., 0:2].transpose(0, 1, 3, 2, 4).reshape(N16, NT, 128)   # d [r, j]
    out[:, :, 1152:] = T[..., 2:4].transpose(0, 1, 3, 2, 4).reshape(N16, NT, 128)       # m [r, j]
    return out.reshape(-1)


def repack_q4_1_loops(q41: np.ndarray) -> np.ndarray:
    N, nb = q41.shape[0], q41.shape[1]
    N16, NT = -(-N // 16), -(-nb // 4)
    out = np.zeros(N16 * NT * 1280, np.uint8)
    for g in range(N16):
        for t in range(NT):
            base = (g * NT + t) * 1280
            for j in range(4):
                for r in range(16):
                    n, b = 16 * g + r, 4 * t + j
                    if n < N and b < nb:
                        out[base + (j * 16 + r) * 16: base + (j * 16 + r) * 16 + 16] = q41[n, b, 4:]
                        out[base + 1024 + (r * 4 + j) * 2: base + 1024 + (r * 4 + j) * 2 + 2] = q41[n, b, 0:2]
                        out[base + 1152 + (r * 4 + j) * 2: base + 1152 + (r * 4 + j) * 2 + 2] = q41[n, b, 2:4]
    return out
