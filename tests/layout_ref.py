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
            lane[:, :, :, :, w, :] = words[:, rows, :, blk, :, :].transpose(0, 2, 1, 3, 4)
        out[:, :, h * 512:(h + 1) * 512] = lane.reshape(N16, NT, 512)
    d = P[..., :2].reshape(N16, 16, NT, 4, 2)                 # [g, row, t, block, 2 bytes]
    sc = np.empty((N16, NT, 8, 4, 2, 2), np.uint8)            # [g, t, r, j, hh, byte]
    for hh in range(2):
        sc[:, :, :, :, hh, :] = d[:, np.arange(8) + 8 * hh].transpose(0, 2, 1, 3, 4)
    out[:, :, 1024:] = sc.reshape(N16, NT, 128)
    return out.reshape(-1)
