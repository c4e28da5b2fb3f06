"""Pins of the CPU oracle to facts outside itself.

Each ``check_*`` function takes an oracle module (the real one, or a mutant
built by ``tests/test_oracle_mutations.py``) and raises AssertionError when the
oracle disagrees with: the hand-worked golden example, brute force from the
raw bytes on tiny shapes, library routines (torch rms_norm / silu / round /
einsum), closed forms, or invariants.  None of them re-types the oracle's own
formula: every check reaches the expected value by another route.
"""

from __future__ import annotations

import os
import random

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            out.setdefault(key, []).append(rest.split())
    return out


def hand_case(fmt: str):
    """(wbuf uint8, x bf16 bits, expected dict) of the hand-worked example."""
    g = read_golden("hand_1x32.txt")
    N, K = int(g["N"][0][0]), int(g["K"][0][0])
    rows = [bytes.fromhex(g[f"{fmt}_row0"][0][0]), bytes.fromhex(g[f"{fmt}_row1"][0][0])]
    rows += [bytes.fromhex(g[f"{fmt}_rest"][0][0])] * (N - 2)
    scales = np.array([float(v) for v in g["scales"][0]], dtype="<f4")
    wbuf = np.frombuffer(b"".join(rows) + scales.tobytes(), dtype=np.uint8).copy()
    x = torch.tensor([[float(v) for v in g["x"][0]]], dtype=torch.float32).to(torch.bfloat16)
    assert torch.equal(x.float(), torch.tensor([[float(v) for v in g["x"][0]]])), "x not exact in bf16"
    xb = x.view(torch.int16).numpy().view(np.uint16)
    exp = {
        "N": N, "K": K, "G": int(g["G"][0][0]),
        "q": np.array([int(v) for v in g["q"][0]], dtype=np.int64),
        "s": float(g["s"][0][0]),
        "acc": np.array([int(v) for v in g["acc"][0]], dtype=np.int64),
        "y": np.array([float(v) for v in g["y"][0]], dtype=np.float32),
    }
    return wbuf, xb, exp


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ----------------------------------------------------------------------------
def check_hand_example(O):
    for fmt in ("w4a8", "w6a8"):
        wbuf, xb, e = hand_case(fmt)
        r = O.forward(fmt, "none", e["N"], e["K"], e["G"], wbuf, x=xb)
        assert np.array_equal(r["q"][0], e["q"]), (fmt, r["q"][0])
        assert r["s"][0] == e["s"], (fmt, r["s"])
        assert np.array_equal(r["acc"][0, :, 0], e["acc"]), (fmt, r["acc"][0, :, 0])
        assert np.array_equal(r["y"][0], e["y"]), (fmt, r["y"][0])


def _bitstream_codes(fmt, N, K, wbuf):
    """Codes read as an LSB-first bit stream per row (independent of the oracle)."""
    b = {"w4a8": 4, "w6a8": 6}[fmt]
    rb = K * b // 8
    out = np.zeros((N, K), dtype=np.int64)
    for n in range(N):
        big = int.from_bytes(bytes(wbuf[n * rb:(n + 1) * rb]), "little")
        for k in range(K):
            out[n, k] = (big >> (b * k)) & ((1 << b) - 1)
    return out


def _bruteforce_y(fmt, N, K, G, wbuf, q, s, codebook=None):
    """y from raw bytes by pure-Python loops over the dequantised weight (levels
    code - offset, or codebook[code])."""
    b = {"w4a8": 4, "w6a8": 6}[fmt]
    codes = _bitstream_codes(fmt, N, K, wbuf)
    off = N * K * b // 8
    scale_bytes = bytes(wbuf[off:off + N * (K // G) * 4])
    sw = [[float(np.frombuffer(scale_bytes[4 * (n * (K // G) + gg):4 * (n * (K // G) + gg) + 4], "<f4")[0])
           for gg in range(K // G)] for n in range(N)]
    M = q.shape[0]
    y = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            tot = 0.0
            for k in range(K):
                lv = float(codebook[int(codes[n, k])]) if codebook is not None else float(int(codes[n, k]) - (1 << (b - 1)))
                w = sw[n][k // G] * lv
                tot += (s[m] * float(q[m, k])) * w
            y[m, n] = tot
    return y


def check_file_layout(O, seed=1):
    rng = np.random.default_rng(seed)
    for fmt in ("w4a8", "w6a8"):
        for (N, K, G) in ((3, 32, 32), (5, 64, 32), (2, 128, 64)):
            nb = N * K * {"w4a8": 4, "w6a8": 6}[fmt] // 8
            wbuf = np.concatenate([rng.integers(0, 256, nb, dtype=np.uint8),
                                   rng.uniform(0.1, 1, N * (K // G)).astype("<f4").view(np.uint8)])
            codes, sw = O.unpack_file(fmt, N, K, G, wbuf)
            assert np.array_equal(codes, _bitstream_codes(fmt, N, K, wbuf)), fmt
            assert np.array_equal(sw.reshape(-1).view(np.uint8), wbuf[nb:]), fmt
            assert np.array_equal(O.pack_file(fmt, codes, sw), wbuf), fmt


def check_forward_bruteforce(O, seed=2):
    rng = random.Random(seed)
    for fmt in ("w4a8", "w6a8"):
        for (N, K, G) in ((16, 32, 32), (16, 64, 32), (32, 128, 64), (16, 128, 32), (16, 64, 16), (32, 96, 16)):
            M = rng.randint(1, 8)
            gen = torch.Generator().manual_seed(rng.randint(0, 10**6))
            x = torch.randn(M, K, generator=gen).to(torch.bfloat16)
            nb = N * K * {"w4a8": 4, "w6a8": 6}[fmt] // 8
            codes = torch.randint(0, 256, (nb,), generator=gen, dtype=torch.uint8).numpy()
            sw = torch.empty(N * (K // G)).uniform_(0.01, 0.02, generator=gen).numpy().astype("<f4")
            wbuf = np.concatenate([codes, sw.view(np.uint8)])
            bias = None
            if rng.random() < 0.5:
                bias = torch.randn(N, generator=gen).numpy().astype(np.float32)
            r = O.forward(fmt, "none", N, K, G, wbuf, x=bits_of(x), bias=bias)
            yb = _bruteforce_y(fmt, N, K, G, wbuf, r["q"], r["s"])
            if bias is not None:
                yb = yb + bias.astype(np.float64)[None, :]
            assert np.allclose(r["y64"], yb, rtol=1e-12, atol=1e-12 * np.abs(yb).max()), (fmt, N, K, G)
    for (N, K, G) in ((16, 32, 8), (16, 64, 4), (32, 96, 8)):  # groups below 16: 4-bit codes only
        gen = torch.Generator().manual_seed(rng.randint(0, 10**6))
        x = torch.randn(3, K, generator=gen).to(torch.bfloat16)
        codes = torch.randint(0, 256, (N * K // 2,), generator=gen, dtype=torch.uint8).numpy()
        sw = torch.empty(N * (K // G)).uniform_(0.01, 0.02, generator=gen).numpy().astype("<f4")
        wbuf = np.concatenate([codes, sw.view(np.uint8)])
        r = O.forward("w4a8", "none", N, K, G, wbuf, x=bits_of(x))
        yb = _bruteforce_y("w4a8", N, K, G, wbuf, r["q"], r["s"])
        assert np.allclose(r["y64"], yb, rtol=1e-12, atol=1e-12 * np.abs(yb).max()), (N, K, G)


def check_quantize(O, seed=3):
    # library route: torch fp32 division and torch.round (ties to even) for the fp32 recipe
    gen = torch.Generator().manual_seed(seed)
    x = (torch.randn(6, 96, generator=gen) * 3).to(torch.bfloat16).float()
    x[2] = 0.0
    x[3] = 0.0
    x[3, 17] = -0.75
    q, s, v = O.quantize_rows(x.double().numpy(), fp32=True)
    amax = x.abs().amax(dim=1)
    st = amax / 127.0
    qt = torch.clamp(torch.round(x / st[:, None]), -127, 127)
    qt[2] = 0
    assert np.array_equal(q, qt[[0, 1, 2, 3, 4, 5]].numpy().astype(np.int64)), "fp32 recipe"
    assert s[2] == 0 and np.all(q[2] == 0), "zero row"
    assert q[3, 17] == -127 and np.count_nonzero(q[3]) == 1, "single nonzero"
    # fp64 route: properties that hold for any correct symmetric RNE quantiser
    a = np.random.default_rng(seed).normal(size=(5, 200)) * np.array([1, 10, 1e-3, 5, 1])[:, None]
    q, s, v = O.quantize_rows(a, fp32=False)
    for m in range(5):
        assert np.isclose(s[m] * 127, np.abs(a[m]).max(), rtol=1e-15)
        assert np.abs(q[m]).max() == 127
        assert np.all(np.abs(q[m] - a[m] / s[m]) <= 0.5 + 1e-12)
    # ties go to even
    t = np.array([[127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5]])
    q, _, _ = O.quantize_rows(t, fp32=False)
    assert list(q[0]) == [127, 0, 2, 2, 0, -2, -2, 126]


def check_prologues(O, seed=4):
    gen = torch.Generator().manual_seed(seed)
    M, K = 3, 256
    x = torch.randn(M, K, generator=gen).to(torch.bfloat16)
    gamma = torch.empty(K).uniform_(0.5, 1.5, generator=gen)
    a = O.prologue("rmsnorm", x=bits_of(x), gamma=gamma.numpy(), eps=1e-6)
    ref = torch.nn.functional.rms_norm(x.double(), (K,), weight=gamma.double(), eps=1e-6)
    assert np.allclose(a, ref.numpy(), rtol=1e-13, atol=0), "rmsnorm vs torch rms_norm"
    g = torch.randn(M, K, generator=gen).to(torch.bfloat16)
    u = torch.randn(M, K, generator=gen).to(torch.bfloat16)
    a = O.prologue("swiglu", gate=bits_of(g), up=bits_of(u))
    ref = torch.nn.functional.silu(g.double()) * u.double()
    assert np.allclose(a, ref.numpy(), rtol=1e-13, atol=1e-300), "swiglu vs torch silu"
    a = O.prologue("none", x=bits_of(x))
    assert np.array_equal(a, x.double().numpy())


def check_closed_forms(O, seed=5):
    rng = np.random.default_rng(seed)
    fmt, N, K, G = "w4a8", 16, 128, 32
    codes = rng.integers(0, 16, (N, K))
    sw = rng.uniform(0.01, 0.02, (N, K // G)).astype(np.float32)
    wbuf = O.pack_file(fmt, codes, sw)
    levels = codes - 8
    deq = np.repeat(sw.astype(np.float64), G, axis=1) * levels          # [N, K]
    # RMSNorm with constant x = c and gamma = 1: a = c / sqrt(c^2 + eps), q = 127 * sign(c)
    for c in (1.5, -0.375, 3.0):
        x = torch.full((1, K), c).to(torch.bfloat16)
        r = O.forward(fmt, "rmsnorm", N, K, G, wbuf, x=bits_of(x), gamma=np.ones(K, np.float32), eps=1e-6)
        a = c / np.sqrt(c * c + 1e-6)
        assert np.all(r["q"] == 127 * np.sign(c))
        assert np.allclose(r["y64"][0], a * deq.sum(axis=1), rtol=1e-12), c
        assert np.array_equal(r["acc"][0], 127 * int(np.sign(c)) * levels.reshape(N, K // G, G).sum(axis=2))
    # SwiGLU with gate = 0 gives 0; with gate = 20, silu(20) = 20 / (1 + e^-20)
    up = torch.randn(2, K, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
    r = O.forward(fmt, "swiglu", N, K, G, wbuf, gate=bits_of(torch.zeros(2, K, dtype=torch.bfloat16)), up=bits_of(up))
    assert np.all(r["y"] == 0) and np.all(r["s"] == 0)
    r = O.forward(fmt, "swiglu", N, K, G, wbuf, gate=bits_of(torch.full((2, K), 20.0, dtype=torch.bfloat16)), up=bits_of(up))
    from scipy.special import expit
    assert np.allclose(r["a"], 20.0 * expit(20.0) * up.double().numpy(), rtol=1e-14)


def check_invariants(O, seed=6):
    rng = np.random.default_rng(seed)
    for fmt in ("w4a8", "w6a8"):
        b = {"w4a8": 4, "w6a8": 6}[fmt]
        N, K, G = 32, 256, 64
        codes = rng.integers(0, 1 << b, (N, K))
        sw = rng.uniform(0.01, 0.02, (N, K // G)).astype(np.float32)
        x = torch.randn(8, K, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
        xb = bits_of(x)
        base = O.forward(fmt, "none", N, K, G, O.pack_file(fmt, codes, sw), x=xb)
        # zero-level codes give 0
        z = O.forward(fmt, "none", N, K, G, O.pack_file(fmt, np.full((N, K), 1 << (b - 1)), sw), x=xb)
        assert np.all(z["y"] == 0) and np.all(z["acc"] == 0)
        # zero scales give 0
        z = O.forward(fmt, "none", N, K, G, O.pack_file(fmt, codes, np.zeros_like(sw)), x=xb)
        assert np.all(z["y"] == 0)
        # doubling every scale doubles y exactly
        d = O.forward(fmt, "none", N, K, G, O.pack_file(fmt, codes, 2 * sw), x=xb)
        assert np.array_equal(d["y64"], 2 * base["y64"])
        # permuting the groups of K together with x leaves y unchanged
        perm = rng.permutation(K // G)
        kperm = (perm[:, None] * G + np.arange(G)[None, :]).reshape(-1)
        p = O.forward(fmt, "none", N, K, G, O.pack_file(fmt, codes[:, kperm], sw[:, perm]), x=xb[:, kperm])
        assert np.allclose(p["y64"], base["y64"], rtol=1e-13, atol=1e-13 * np.abs(base["y64"]).max())
        # rows are independent: row m of the 8-row call equals the 1-row call
        for m in (0, 5, 7):
            one = O.forward(fmt, "none", N, K, G, O.pack_file(fmt, codes, sw), x=xb[m:m + 1])
            assert np.array_equal(one["y"][0], base["y"][m])
        # group sums agree with an int64 einsum (library route)
        acc = np.einsum("mgk,ngk->mng", base["q"].reshape(8, K // G, G), (codes - (1 << (b - 1))).reshape(N, K // G, G))
        assert np.array_equal(acc, base["acc"])


def check_stream_positions(O):
    g = read_golden("stream_positions.txt")
    N, K, G = 16, 32, 32
    rows = [[int(key)] + [int(v) for v in rest] for key in ("0", "9", "3", "15") for rest in g[key]]
    for fmt in ("w4a8", "w6a8"):
        size = O.file_bytes(fmt, N, K, G)
        for n, k, nb, ns, hb, hs in rows:
            buf = np.zeros(size, dtype=np.uint8)
            buf[nb] = 0x5 << ns
            if fmt == "w6a8":
                buf[hb] = 0x2 << hs
            codes, _ = O.unpack_stream(fmt, N, K, G, buf)
            want = np.zeros((N, K), dtype=np.int64)
            want[n, k] = 5 + (32 if fmt == "w6a8" else 0)
            assert np.array_equal(codes, want), (fmt, n, k, np.argwhere(codes))
        # scale order within the scale block
        buf = np.zeros(size, dtype=np.uint8)
        buf[:64] = np.arange(16, dtype="<f4").view(np.uint8)
        _, sw = O.unpack_stream(fmt, N, K, G, buf)
        for slot, row in enumerate(int(v) for v in g["scale_rows"][0]):
            assert sw[row, 0] == slot, (fmt, row, sw[:, 0])


def check_stream_bijection(O):
    """Every code is read from its own field of the stream, and no two codes share one.

    Each byte p of the buffer is labelled with its index, one 4-bit (or 2-bit)
    digit at a time, by writing the digit into every field of the byte; the
    unpacked code at (n, k) then reports the digit of the byte it came from.
    Ragged tile (N % 128 != 0), several units, and G > 128 are covered."""
    for fmt, N, K, G in (("w4a8", 144, 160, 32), ("w6a8", 144, 160, 32), ("w4a8", 32, 256, 256), ("w6a8", 16, 512, 256)):
        size = O.file_bytes(fmt, N, K, G)
        assert size < (1 << 16)
        p = np.arange(size)
        src = np.zeros((N, K), dtype=np.int64)
        for j in range(4):
            d = ((p >> (4 * j)) & 0xF).astype(np.uint8)
            codes, _ = O.unpack_stream(fmt, N, K, G, d | (d << 4))
            src |= (codes & 0xF) << (4 * j)
        half, _ = O.unpack_stream(fmt, N, K, G, np.full(size, 0x10, dtype=np.uint8))
        key = src * 2 + ((half & 0xF) >> 0)      # 0 = low nibble, 1 = high nibble
        assert np.unique(key).size == N * K, fmt
        if fmt == "w6a8":
            hsrc = np.zeros((N, K), dtype=np.int64)
            for j in range(8):
                d = ((p >> (2 * j)) & 0x3).astype(np.uint8)
                codes, _ = O.unpack_stream(fmt, N, K, G, d * np.uint8(0x55))
                hsrc |= (codes >> 4) << (2 * j)
            slot, _ = O.unpack_stream(fmt, N, K, G, np.full(size, 0b11100100, dtype=np.uint8))
            hkey = hsrc * 4 + (slot >> 4)
            assert np.unique(hkey).size == N * K, fmt
            assert not np.intersect1d(src, hsrc).size, "2-bit plane shares bytes with the 4-bit plane"


def check_stream_positions_codebook(O):
    """The codebook layout: single codes at hand-derived positions, and every
    code read from its own field (bijection), ragged tile and several units
    included."""
    g = read_golden("stream_positions_codebook.txt")
    N, K, G = 16, 32, 32
    size = O.file_bytes("w4a8", N, K, G)
    for key in ("0", "9", "3", "15"):
        for rest in g[key]:
            n, k, nb, ns = int(key), int(rest[0]), int(rest[1]), int(rest[2])
            buf = np.zeros(size, dtype=np.uint8)
            buf[nb] = 0x5 << ns
            codes, _ = O.unpack_stream("w4a8", N, K, G, buf, layout="codebook")
            want = np.zeros((N, K), dtype=np.int64)
            want[n, k] = 5
            assert np.array_equal(codes, want), (n, k, np.argwhere(codes))
    for N, K, G in ((144, 160, 32), (32, 256, 256)):
        size = O.file_bytes("w4a8", N, K, G)
        p = np.arange(size)
        src = np.zeros((N, K), dtype=np.int64)
        for j in range(4):
            d = ((p >> (4 * j)) & 0xF).astype(np.uint8)
            codes, _ = O.unpack_stream("w4a8", N, K, G, d | (d << 4), layout="codebook")
            src |= (codes & 0xF) << (4 * j)
        half, _ = O.unpack_stream("w4a8", N, K, G, np.full(size, 0x10, dtype=np.uint8), layout="codebook")
        key = src * 2 + (half & 0xF)
        assert np.unique(key).size == N * K


def check_stream_positions_rows(O):
    """The row layout: single codes at hand-derived positions (both formats),
    the scale order, and every code read from its own field (bijection) on a
    ragged tile, several units and G > 128."""
    g = read_golden("stream_positions_rows.txt")
    N, K, G = 16, 32, 32
    rows = [[int(key)] + [int(v) for v in rest] for key in ("0", "9", "3", "15", "5") for rest in g[key]]
    for fmt in ("w4a8", "w6a8"):
        size = O.file_bytes(fmt, N, K, G)
        for n, k, nb, ns, hb, hs in rows:
            buf = np.zeros(size, dtype=np.uint8)
            buf[nb] = 0x5 << ns
            if fmt == "w6a8":
                buf[hb] = 0x2 << hs
            codes, _ = O.unpack_stream(fmt, N, K, G, buf, layout="rows")
            want = np.zeros((N, K), dtype=np.int64)
            want[n, k] = 5 + (32 if fmt == "w6a8" else 0)
            assert np.array_equal(codes, want), (fmt, n, k, np.argwhere(codes))
        buf = np.zeros(size, dtype=np.uint8)
        buf[:64] = np.arange(16, dtype="<f4").view(np.uint8)
        _, sw = O.unpack_stream(fmt, N, K, G, buf, layout="rows")
        for slot, row in enumerate(int(v) for v in g["scale_rows"][0]):
            assert sw[row, 0] == slot, (fmt, row, sw[:, 0])
        # two chunks and two groups in one unit: chunk-major planes, [group][row] scales
        n, k, nb, ns, hb, hs = (int(v) for v in g["wide"][0])
        size = O.file_bytes(fmt, 16, 64, 32)
        buf = np.zeros(size, dtype=np.uint8)
        buf[nb] = 0x5 << ns
        if fmt == "w6a8":
            buf[hb] = 0x2 << hs
        codes, _ = O.unpack_stream(fmt, 16, 64, 32, buf, layout="rows")
        want = np.zeros((16, 64), dtype=np.int64)
        want[n, k] = 5 + (32 if fmt == "w6a8" else 0)
        assert np.array_equal(codes, want), (fmt, n, k, np.argwhere(codes))
        row, grp, byte = (int(v) for v in g["wide_scale"][0])
        buf = np.zeros(size, dtype=np.uint8)
        buf[byte:byte + 4] = np.array([7.0], dtype="<f4").view(np.uint8)
        _, sw = O.unpack_stream(fmt, 16, 64, 32, buf, layout="rows")
        assert sw[row, grp] == 7.0 and np.count_nonzero(sw) == 1, (fmt, np.argwhere(sw))
    for fmt, N, K, G in (("w4a8", 144, 160, 32), ("w6a8", 144, 160, 32), ("w4a8", 32, 512, 256), ("w6a8", 16, 384, 64)):
        size = O.file_bytes(fmt, N, K, G)
        assert size < (1 << 16)
        p = np.arange(size)
        src = np.zeros((N, K), dtype=np.int64)
        for j in range(4):
            d = ((p >> (4 * j)) & 0xF).astype(np.uint8)
            codes, _ = O.unpack_stream(fmt, N, K, G, d | (d << 4), layout="rows")
            src |= (codes & 0xF) << (4 * j)
        half, _ = O.unpack_stream(fmt, N, K, G, np.full(size, 0x10, dtype=np.uint8), layout="rows")
        key = src * 2 + (half & 0xF)
        assert np.unique(key).size == N * K, fmt
        if fmt == "w6a8":
            hsrc = np.zeros((N, K), dtype=np.int64)
            for j in range(8):
                d = ((p >> (2 * j)) & 0x3).astype(np.uint8)
                codes, _ = O.unpack_stream(fmt, N, K, G, d * np.uint8(0x55), layout="rows")
                hsrc |= (codes >> 4) << (2 * j)
            slot, _ = O.unpack_stream(fmt, N, K, G, np.full(size, 0b11100100, dtype=np.uint8), layout="rows")
            hkey = hsrc * 4 + (slot >> 4)
            assert np.unique(hkey).size == N * K, fmt
            assert not np.intersect1d(src, hsrc).size, "2-bit plane shares bytes with the 4-bit plane"


def check_bias(O, seed=9):
    """A float bias is added once, unscaled, to every row: with every level zero
    y equals the bias exactly; sampled columns take the matching entries."""
    rng = np.random.default_rng(seed)
    for fmt in ("w4a8", "w6a8"):
        b = {"w4a8": 4, "w6a8": 6}[fmt]
        N, K, G = 32, 128, 32
        bias = rng.normal(size=N).astype(np.float32) * 3
        sw = rng.uniform(0.01, 0.02, (N, K // G)).astype(np.float32)
        x = torch.randn(3, K, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
        zero = O.pack_file(fmt, np.full((N, K), 1 << (b - 1)), sw)
        r = O.forward(fmt, "none", N, K, G, zero, x=bits_of(x), bias=bias)
        assert np.array_equal(r["y"], np.broadcast_to(bias, (3, N))), fmt
        codes = rng.integers(0, 1 << b, (N, K))
        wbuf = O.pack_file(fmt, codes, sw)
        full = O.forward(fmt, "rmsnorm", N, K, G, wbuf, x=bits_of(x), gamma=np.ones(K, np.float32), bias=bias)
        cols = np.array([0, 5, 17, 31])
        part = O.forward(fmt, "rmsnorm", N, K, G, wbuf, x=bits_of(x), gamma=np.ones(K, np.float32), bias=bias,
                         cols=cols)
        assert np.array_equal(part["y64"], full["y64"][:, cols]), fmt


def check_moe(O, seed=10):
    """An expert bank is E separate weights stacked along the output rows:
    each routed (token, slot) equals a plain forward of that expert's own
    weight (packed on its own) for that token alone, bias included; a token
    routed to one expert twice gets the same rows in both slots."""
    rng = np.random.default_rng(seed)
    for fmt in ("w4a8", "w6a8"):
        b = {"w4a8": 4, "w6a8": 6}[fmt]
        E, N, K, G = 5, 32, 64, 32
        codes = rng.integers(0, 1 << b, (E * N, K))
        sw = rng.uniform(0.01, 0.02, (E * N, K // G)).astype(np.float32)
        bias = rng.normal(size=(E, N)).astype(np.float32)
        bank = O.pack_file(fmt, codes, sw)
        x = torch.randn(3, K, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
        gamma = rng.uniform(0.5, 1.5, K).astype(np.float32)
        ids = np.array([[4, 1], [0, 0], [2, 4]])
        r = O.forward_moe(fmt, "rmsnorm", E, N, K, G, bank, ids, x=bits_of(x), gamma=gamma, bias=bias)
        for m in range(3):
            for j in range(2):
                e = ids[m, j]
                own = O.pack_file(fmt, codes[e * N:(e + 1) * N], sw[e * N:(e + 1) * N])
                one = O.forward(fmt, "rmsnorm", N, K, G, own, x=bits_of(x[m:m + 1]), gamma=gamma, bias=bias[e])
                assert np.array_equal(r["y64"][m, j], one["y64"][0]), (fmt, m, j)
        assert np.array_equal(r["y64"][1, 0], r["y64"][1, 1])


def check_codebook(O, seed=11):
    """A 4-bit codebook replaces the uniform levels: the uniform table
    (c - 8) gives back the plain result exactly, and any table matches the
    brute-force dequantised product."""
    rng = np.random.default_rng(seed)
    N, K, G = 16, 64, 32
    codes = rng.integers(0, 16, (N, K))
    sw = rng.uniform(0.01, 0.02, (N, K // G)).astype(np.float32)
    wbuf = O.pack_file("w4a8", codes, sw)
    x = torch.randn(3, K, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
    plain = O.forward("w4a8", "none", N, K, G, wbuf, x=bits_of(x))
    uni = O.forward("w4a8", "none", N, K, G, wbuf, x=bits_of(x), codebook=np.arange(16, dtype=np.float32) - 8)
    assert np.array_equal(plain["y64"], uni["y64"])
    cb = np.sort(rng.normal(size=16)).astype(np.float32)  # an NF4-like, non-uniform table
    r = O.forward("w4a8", "rmsnorm", N, K, G, wbuf, x=bits_of(x), gamma=np.ones(K, np.float32), codebook=cb)
    yb = _bruteforce_y("w4a8", N, K, G, wbuf, r["q"], r["s"], codebook=cb)
    assert np.allclose(r["y64"], yb, rtol=1e-12, atol=1e-12 * np.abs(yb).max())



def check_float_sanity(O, seed=12):
    """The quantised result against the unquantised fp64 product of the
    prologue output and the dequantised weight ("Comfy Quantization Formats",
    section "Activations and smoothing": a backend without the integer kernel
    dequantises and runs the float linear).  Everything on the float side is
    computed independently of the oracle: the prologue with torch (rms_norm,
    silu), the weight from the raw bytes through the bit-stream reader.  Per-row
    symmetric int8 quantisation moves each activation by at most s_m / 2 with
    s_m = amax_m / 127, so |y - y_float| <= s_m / 2 * sum_k |w[n, k]| exactly;
    a wrong sign, offset, scale or prologue breaks the bound."""
    rng = np.random.default_rng(seed)
    for fmt in ("w4a8", "w6a8"):
        b = {"w4a8": 4, "w6a8": 6}[fmt]
        N, K, G = 16, 96, 32
        codes = rng.integers(0, 1 << b, (N, K))
        sw = rng.uniform(0.01, 0.02, (N, K // G)).astype(np.float32)
        wbuf = O.pack_file(fmt, codes, sw)
        raw = _bitstream_codes(fmt, N, K, wbuf) - (1 << (b - 1))
        w = np.repeat(np.frombuffer(bytes(wbuf[N * K * b // 8:]), "<f4").reshape(N, K // G).astype(np.float64),
                      G, axis=1) * raw
        gen = torch.Generator().manual_seed(seed)
        x = torch.randn(4, K, generator=gen).to(torch.bfloat16)
        g = torch.randn(4, K, generator=gen).to(torch.bfloat16)
        u = torch.randn(4, K, generator=gen).to(torch.bfloat16)
        gamma = torch.empty(K).uniform_(0.5, 1.5, generator=gen)
        cases = {
            "none": (x.double(), dict(x=bits_of(x))),
            "rmsnorm": (torch.nn.functional.rms_norm(x.double(), (K,), weight=gamma.double(), eps=1e-6),
                        dict(x=bits_of(x), gamma=gamma.numpy(), eps=1e-6)),
            "swiglu": (torch.nn.functional.silu(g.double()) * u.double(), dict(gate=bits_of(g), up=bits_of(u))),
        }
        for kind, (a, kw) in cases.items():
            a = a.numpy()
            r = O.forward(fmt, kind, N, K, G, wbuf, **kw)
            yf = a @ w.T
            s = np.abs(a).max(axis=1) / 127.0
            bound = (s / 2.0)[:, None] * np.abs(w).sum(axis=1)[None, :]
            err = np.abs(r["y64"] - yf)
            assert np.all(err <= bound * (1 + 1e-9) + 1e-12), (fmt, kind, float((err / bound).max()))
            # and the bound is not vacuous: the error is a small fraction of y
            assert float(err.max()) < 0.05 * float(np.abs(yf).max()), (fmt, kind)
