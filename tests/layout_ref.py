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
    words = P[..., 2:].reshape(N16, 16, NT, 4, 4, 4)        # [g, row, t, block, c, byte]
    out = np.zeros((N16, NT, 1152), np.uint8)
    for h in range(2):
        # [g, t, r, c, word, byte] for the 32 lanes L = 4r + c
        lane = np.empty((N16, NT, 8, 4, 4, 4), np.uint8)
        for w in range(4):
            rows = np.arange(8) + 8 * (w % 2)
            blk = 2 * h + w // 2
            lane[:, :, :, :, w, :] = words[:, rows][:, :, :, blk].transpose(0, 2, 1, 3, 4)
        out[:, :, h * 512:(h + 1) * 512] = lane.reshape(N16, NT, 512)
    d = P[..., :2].reshape(N16, 16, NT, 4, 2)                 # [g, row, t, block, 2 bytes]
    sc = np.empty((N16, NT, 8, 4, 2, 2), np.uint8)            # [g, t, r, j, hh, byte]
    for hh in range(2):
        sc[:, :, :, :, hh, :] = d[:, np.arange(8) + 8 * hh].transpose(0, 2, 1, 3, 4)
    out[:, :, 1024:] = sc.reshape(N16, NT, 128)
    return out.reshape(-1)


def repack_loops(q4: np.ndarray) -> np.ndarray:
    """The same layout, byte by byte, in the words of the header (slow; small sizes)."""
    N, nb = q4.shape[0], q4.shape[1]
    N16, NT = -(-N // 16), -(-nb // 4)
    out = np.zeros(N16 * NT * 1152, np.uint8)

    def code_byte(n, b, i):
        return q4[n, b, 2 + i] if (n < N and b < nb) else 0x88

    def scale_byte(n, b, i):
        return q4[n, b, i] if (n < N and b < nb) else 0

    for g in range(N16):
        for t in range(NT):
            base = (g * NT + t) * 1152
            for h in range(2):
                for L in range(32):
                    r, c = L // 4, L % 4
                    srcs = [(16 * g + r, 4 * t + 2 * h), (16 * g + r + 8, 4 * t + 2 * h),
                            (16 * g + r, 4 * t + 2 * h + 1), (16 * g + r + 8, 4 * t + 2 * h + 1)]
                    for w, (n, b) in enumerate(srcs):
                        for i in range(4):
                            out[base + h * 512 + L * 16 + 4 * w + i] = code_byte(n, b, 4 * c + i)
            for r in range(8):
                k = 0
                for j in range(4):
                    for n in (16 * g + r, 16 * g + r + 8):
                        for i in range(2):
                            out[base + 1024 + r * 16 + k] = scale_byte(n, 4 * t + j, i)
                            k += 1
    return out
