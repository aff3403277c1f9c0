"""Small shared helpers for the tests (no method arithmetic)."""
import numpy as np
import torch


def bf16(a):
    import synth
    return synth.to_bf16_bits(np.asarray(a, np.float32))


def f32(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def torch_bf16(x32):
    return torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


E4M3_POS = np.array([2.0 ** e * (1 + m / 8) for e in range(-6, 9) for m in range(8)
                     if 2.0 ** e * (1 + m / 8) <= 448])
E2M1_SIGNED = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -1.5, -2, -3, -4, -6])


def lossless_rows(rng, rows, K, g_exp):
    """Rows x = g s_b c with power-of-two g: block 0 has scale 448 and holds
    the row amax 6*448*g, every other block holds 6 s_b g, so every quotient
    of the quantiser is exact and the NVFP4 encoding is lossless."""
    g = 2.0 ** g_exp
    x = np.zeros((rows, K))
    for r in range(rows):
        for b in range(K // 16):
            s = 448.0 if b == 0 else rng.choice(E4M3_POS)
            blk = rng.choice(E2M1_SIGNED, 16)
            blk[rng.integers(16)] = 6.0 * rng.choice([1, -1])
            x[r, b * 16:(b + 1) * 16] = blk * s * g
    return x.astype(np.float32)
