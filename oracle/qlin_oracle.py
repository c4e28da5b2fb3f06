"""CPU oracle for the skinny W4A8 / W6A8 quantized linear.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module. The product path (``w6a8_quantized_linear_gb300``) never does, and this
module imports nothing from it: the two share no code.

What it computes is the plain definition of the method, written out step by
step in float64 / int64 with numpy:

1. unpack the checkpoint ("file") layout into integer codes and fp32 group
   scales                                    -- ``unpack_file``
2. the prologue: none, RMSNorm or SwiGLU     -- ``prologue``
3. per-row symmetric int8 quantisation       -- ``quantize_rows``
4. per-group integer dot products            -- ``group_acc``
5. y = s_m * sum_g sw[n,g] * acc[m,n,g]      -- ``forward``
   (+ bias[n] when the layer has a float bias)

plus ``unpack_stream``, an independent reading of the kernel-order stream
layout that the in-place repack produces (used to check the GPU repack byte
for byte).

Sources (page title, section):

* "Doubling the LLM token rate in ComfyUI" (ComfyUI blog), section
  "Optimising the linear kernel": decode is a skinny product of a dense weight
  with M = 1 (or a few MTP rows, up to 8); W4A8 / W6A8 checkpoints; the
  activations are quantised to int8 inside the linear kernel; weights and their
  per-group scales are interleaved in the order the kernel reads them, by a
  one-time in-place repack; the activation quantisation absorbs the RMSNorm or
  SwiGLU in front of it.
* "Comfy Quantization Formats", section "Weight formats": N is the output
  width, K the input width, G the group size, scales are FP32.
* same page, section "Format options": ``asym_w4a8_int8`` uses uniform levels
  when it has no codebook, ``w6a8_int8`` has none, weights are symmetric;
  shape rules for K and G.
* same page, section "Activations and smoothing": integer formats take float
  input and quantise activations inside the kernel, with no stored input scale;
  biases stay floating point (section "Checkpoint layout": an ordinary float
  bias beside the quantised weight, if present).

Readings where the pages are silent (each is listed in the design notes):

* level = code - 2**(b-1) (8 for 4-bit, 32 for 6-bit); no zero point.
* file layout, LSB-first bit stream per row: 4-bit: uint8 [N, K/2], low nibble
  holds the even k; 6-bit: uint8 [N, 3K/4], every 3 bytes hold 4 codes as a
  little-endian 24-bit word, code i at bits 6i..6i+5. fp32 scales [N, K/G]
  (row-major, little-endian) follow the codes in the same buffer.
* scale s = amax/127, q = clamp(round-half-even(a/s), -127, 127); an all-zero
  row gives s = 0 and q = 0.
* with no prologue the quantisation is taken in fp32 (s = fl32(amax/127),
  v = fl32(x/s)), the precision the kernel uses, so that codes are unique;
  with a prologue it is taken in fp64 from the fp64 prologue value.
* RMSNorm: a = x * gamma / sqrt(mean(x^2) + eps), gamma used as given.
* SwiGLU: a = silu(gate) * up = gate / (1 + exp(-gate)) * up.

Every function below is pinned by tests in ``tests/test_oracle.py`` against a
hand-worked example, brute force on tiny shapes, closed forms, library
routines and invariants; no function is "parity unpinned".
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "BITS", "code_offset", "file_code_bytes", "file_scale_bytes", "file_bytes",
    "unpack_file", "pack_file", "bf16_bits_to_f64", "prologue", "quantize_rows",
    "group_acc", "group_acc_codebook", "forward", "forward_moe", "STREAM_TN", "stream_kb", "unpack_stream",
]

BITS = {"w4a8": 4, "w6a8": 6}


def code_offset(fmt: str) -> int:
    """Zero level of the uniform symmetric grid: level = code - 2**(b-1).

    Reading of "Comfy Quantization Formats", section "Format options"
    (uniform levels, symmetric export)."""
    return 1 << (BITS[fmt] - 1)


def file_code_bytes(fmt: str, N: int, K: int) -> int:
    return N * K * BITS[fmt] // 8


def file_scale_bytes(N: int, K: int, G: int) -> int:
    return N * (K // G) * 4


def file_bytes(fmt: str, N: int, K: int, G: int) -> int:
    return file_code_bytes(fmt, N, K) + file_scale_bytes(N, K, G)


# ----------------------------------------------------------------------------
# 1. checkpoint layout
# ----------------------------------------------------------------------------

def unpack_file(fmt: str, N: int, K: int, G: int, buf, rows=None) -> tuple[np.ndarray, np.ndarray]:
    """Split a checkpoint-layout buffer into codes int64 [N, K] and fp32 scales [N, K/G].

    ``rows`` (optional) selects output rows n to unpack, for sampled checks.
    "Comfy Quantization Formats", section "Weight formats" (N, K, G, FP32
    scales); bit order per the reading in the module docstring."""
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    ncb = file_code_bytes(fmt, N, K)
    assert buf.size >= file_bytes(fmt, N, K, G)
    N_all = N
    rows = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    cb = buf[:ncb].reshape(N, K * BITS[fmt] // 8)[rows].astype(np.int64)
    N = rows.size
    codes = np.empty((N, K), dtype=np.int64)
    if BITS[fmt] == 4:
        codes[:, 0::2] = cb & 0xF
        codes[:, 1::2] = cb >> 4
    else:
        t = cb.reshape(N, K // 4, 3)
        word = t[..., 0] | (t[..., 1] << 8) | (t[..., 2] << 16)
        for i in range(4):
            codes[:, i::4] = (word >> (6 * i)) & 0x3F
    sw = np.frombuffer(buf[ncb:ncb + file_scale_bytes(N_all, K, G)].tobytes(), dtype="<f4")
    return codes, sw.reshape(N_all, K // G)[rows].astype(np.float32)


def pack_file(fmt: str, codes, sw) -> np.ndarray:
    """Inverse of ``unpack_file``: codes int [N, K] in [0, 2**b) and scales [N, K/G]."""
    codes = np.asarray(codes, dtype=np.int64)
    N, K = codes.shape
    assert codes.min() >= 0 and codes.max() < (1 << BITS[fmt])
    if BITS[fmt] == 4:
        cb = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    else:
        word = np.zeros((N, K // 4), dtype=np.int64)
        for i in range(4):
            word |= codes[:, i::4] << (6 * i)
        cb = np.stack([word & 0xFF, (word >> 8) & 0xFF, (word >> 16) & 0xFF], axis=-1).astype(np.uint8)
    sb = np.ascontiguousarray(np.asarray(sw, dtype="<f4")).view(np.uint8)
    return np.concatenate([cb.reshape(-1), sb.reshape(-1)])


# ----------------------------------------------------------------------------
# 2. prologue
# ----------------------------------------------------------------------------

def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def prologue(kind: str, x=None, gate=None, up=None, gamma=None, eps: float = 1e-6) -> np.ndarray:
    """Activation a [M, K] in float64 from bf16 inputs (given as uint16 bits).

    "Doubling the LLM token rate in ComfyUI", section "Optimising the linear
    kernel": the quantisation absorbs the RMSNorm or the SwiGLU before it.
    """
    if kind == "none":
        return bf16_bits_to_f64(x)
    if kind == "rmsnorm":
        xv = bf16_bits_to_f64(x)
        K = xv.shape[1]
        g = np.asarray(gamma, dtype=np.float32).astype(np.float64)
        mean_sq = (xv * xv).sum(axis=1) / K
        return xv * g[None, :] / np.sqrt(mean_sq + float(eps))[:, None]
    if kind == "swiglu":
        gv = bf16_bits_to_f64(gate)
        uv = bf16_bits_to_f64(up)
        with np.errstate(over="ignore"):
            return gv / (1.0 + np.exp(-gv)) * uv
    raise ValueError(kind)


# ----------------------------------------------------------------------------
# 3. per-row int8 quantisation
# ----------------------------------------------------------------------------

def quantize_rows(a, fp32: bool) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Per-row symmetric int8 quantisation of a [M, K].

    s_m = max_k |a[m,k]| / 127, q = clamp(round_half_even(a / s_m), -127, 127),
    s_m = 0 and q = 0 for an all-zero row.  With ``fp32`` the two divisions are
    taken in IEEE fp32 (numpy float32 arithmetic is correctly rounded); else in
    float64.  Returns (q int64 [M,K], s float64 [M], v float64 [M,K]) where v is
    the value that was rounded (a/s), kept for the rounding-boundary rule.

    "Comfy Quantization Formats", section "Activations and smoothing" (dynamic
    in-kernel activation quantisation, no stored input scale).
    """
    a = np.asarray(a, dtype=np.float64)
    M, K = a.shape
    q = np.zeros((M, K), dtype=np.int64)
    s = np.zeros(M, dtype=np.float64)
    v = np.zeros((M, K), dtype=np.float64)
    for m in range(M):
        if fp32:
            row = a[m].astype(np.float32)
            assert np.array_equal(row.astype(np.float64), a[m]), "fp32 recipe needs fp32-exact inputs"
            amax = np.float32(np.abs(row).max()) if K else np.float32(0)
            if amax == 0:
                continue
            sm = np.float32(amax / np.float32(127.0))
            vm = (row / sm).astype(np.float32)
            s[m] = float(sm)
            v[m] = vm.astype(np.float64)
        else:
            amax = float(np.abs(a[m]).max()) if K else 0.0
            if amax == 0.0:
                continue
            s[m] = amax / 127.0
            v[m] = a[m] / s[m]
        q[m] = np.clip(np.rint(v[m]), -127, 127).astype(np.int64)  # np.rint: ties to even
    return q, s, v


# ----------------------------------------------------------------------------
# 4. per-group integer dot products
# ----------------------------------------------------------------------------

def group_acc(q, codes, fmt: str, G: int) -> np.ndarray:
    """acc[m, n, g] = sum_{k in group g} q[m, k] * (codes[n, k] - offset), int64.

    The contraction is done as a float64 matmul per group: every product is an
    integer of magnitude <= 127 * 32 and every partial sum is below 2**53, so
    the float64 result is the exact integer; this is asserted.

    "Doubling the LLM token rate in ComfyUI", section "Optimising the linear
    kernel" (the MMA computes integer dot products of int8 activations with the
    weight levels, one accumulator per scale group)."""
    q = np.asarray(q, dtype=np.int64)
    L = np.asarray(codes, dtype=np.int64) - code_offset(fmt)
    M, K = q.shape
    N = L.shape[0]
    ng = K // G
    qg = q.reshape(M, ng, G).transpose(1, 0, 2).astype(np.float64)      # [g, M, G]
    Lg = L.reshape(N, ng, G).transpose(1, 2, 0).astype(np.float64)      # [g, G, N]
    acc = np.matmul(qg, Lg)                                              # [g, M, N]
    acc_i = np.rint(acc).astype(np.int64)
    assert np.array_equal(acc_i.astype(np.float64), acc)
    return acc_i.transpose(1, 2, 0)                                      # [M, N, g]


def group_acc_codebook(q, codes, codebook, G: int) -> np.ndarray:
    """acc[m, n, g] = sum_{k in group g} q[m, k] * codebook[codes[n, k]], float64.

    "Comfy Quantization Formats", section "Format options": an asym_w4a8_int8
    weight may store a float [16] weight_codebook that replaces the uniform
    levels (code - 8).  Reading: the level of code c is codebook[c] (fp32),
    one table per weight; the sums are no longer integers."""
    q = np.asarray(q, dtype=np.float64)
    L = np.asarray(codebook, dtype=np.float32).astype(np.float64)[np.asarray(codes)]
    M, K = q.shape
    N = L.shape[0]
    ng = K // G
    qg = q.reshape(M, ng, G).transpose(1, 0, 2)                          # [g, M, G]
    Lg = L.reshape(N, ng, G).transpose(1, 2, 0)                          # [g, G, N]
    return np.matmul(qg, Lg).transpose(1, 2, 0)                          # [M, N, g]


# ----------------------------------------------------------------------------
# 5. the whole path
# ----------------------------------------------------------------------------

def forward(fmt: str, kind: str, N: int, K: int, G: int, buf, x=None, gate=None, up=None,
            gamma=None, eps: float = 1e-6, cols=None, stream: bool = False, bias=None, codebook=None) -> dict:
    """y[M, N] = s_m * sum_g sw[n, g] * acc[m, n, g] (+ bias[n]), in float64,
    rounded to fp32.  ``bias`` is an optional fp32 [N] vector (reading: an
    ordinary float bias is added after the scaled product).  ``codebook`` is
    an optional fp32 [16] table of levels for 4-bit codes (``acc`` is then
    float64 rather than integer).

    ``buf`` is the checkpoint layout (or, with ``stream=True``, the repacked
    stream layout).  ``cols`` restricts the computation to the listed output
    columns n (for sampled checks at full size).  Returns a dict with
    y (fp32), y64, q, s, v and acc.
    """
    if stream:
        codes, sw = unpack_stream(fmt, N, K, G, buf)
        if cols is not None:
            codes, sw = codes[cols], sw[cols]
    else:
        codes, sw = unpack_file(fmt, N, K, G, buf, rows=cols)
    a = prologue(kind, x=x, gate=gate, up=up, gamma=gamma, eps=eps)
    q, s, v = quantize_rows(a, fp32=(kind == "none"))
    if codebook is not None:
        assert fmt == "w4a8", "only 4-bit codes have a codebook"
        acc = group_acc_codebook(q, codes, codebook, G)
    else:
        acc = group_acc(q, codes, fmt, G)
    y64 = s[:, None] * (acc.astype(np.float64) * sw.astype(np.float64)[None, :, :]).sum(axis=2)
    if bias is not None:
        b = np.asarray(bias, dtype=np.float32).astype(np.float64)
        y64 = y64 + (b if cols is None else b[np.asarray(cols)])[None, :]
    return {"y": y64.astype(np.float32), "y64": y64, "q": q, "s": s, "v": v, "acc": acc, "a": a}


def forward_moe(fmt: str, kind: str, E: int, N: int, K: int, G: int, bank, ids, x=None, gate=None, up=None,
                gamma=None, eps: float = 1e-6, bias=None, rows=None) -> dict:
    """Expert bank: y[m, j, :] = expert ids[m, j] applied to token m.

    "Comfy Quantization Formats", section "Embeddings and MoE": an expert
    bank's weights and per-expert scales carry a leading expert dimension E;
    a grouped W4A8 / W6A8 bank may be stored with expert and output rows
    flattened to E * N (so ``bank`` is the checkpoint layout of an [E * N, K]
    weight); the optional bias is [E, N].  Readings: every token is
    quantised once, as for a plain linear; ids [M, topk] selects, for each
    token, the experts whose outputs are returned (no routing weights are
    applied).  ``rows`` limits the check to listed output rows n < N.
    Returns y [M, topk, N'] (float64 and fp32) and the token codes.
    """
    ids = np.asarray(ids, dtype=np.int64)
    M, topk = ids.shape
    sel = np.arange(N) if rows is None else np.asarray(rows)
    used = sorted(set(int(e) for e in ids.ravel()))
    y64 = np.zeros((M, topk, sel.size))
    q = s = None
    for e in used:
        cols = e * N + sel
        r = forward(fmt, kind, E * N, K, G, bank, x=x, gate=gate, up=up, gamma=gamma, eps=eps, cols=cols,
                    bias=None if bias is None else np.asarray(bias, np.float32).reshape(E * N))
        q, s = r["q"], r["s"]
        for m in range(M):
            for j in range(topk):
                if ids[m, j] == e:
                    y64[m, j] = r["y64"][m]
    return {"y": y64.astype(np.float32), "y64": y64, "q": q, "s": s}


# ----------------------------------------------------------------------------
# the kernel-order stream (output of the in-place repack)
# ----------------------------------------------------------------------------

STREAM_TN = 128  # output rows per tile


def stream_kb(G: int) -> int:
    """k extent of one stream unit: max(128, G)."""
    return max(128, G)


def _slab_pair_index():
    """Row-in-slab and k-in-pair of every (lane, step, register, element) of one
    16-row x 32-k piece of the code block.

    A-operand registers of lane (g, t) of a 16x16 bf16 tensor-core tile hold
    (row g, k 2t..2t+1), (row g+8, k 2t..2t+1), (row g, k 2t+8..2t+9),
    (row g+8, k 2t+8..2t+9); step B is step A shifted by 16 in k."""
    lane = np.arange(32)[:, None, None, None]
    step = np.arange(2)[None, :, None, None]
    reg = np.arange(4)[None, None, :, None]
    elem = np.arange(2)[None, None, None, :]
    g, t = lane // 4, lane % 4
    row = g + 8 * (reg % 2)
    kk = 16 * step + 2 * t + 8 * (reg // 2) + elem
    return np.broadcast_to(row, (32, 2, 4, 2)), np.broadcast_to(kk, (32, 2, 4, 2))


def unpack_stream(fmt: str, N: int, K: int, G: int, buf, layout: str = "plain") -> tuple[np.ndarray, np.ndarray]:
    """Read codes [N, K] and scales [N, K/G] back out of the stream layout.

    The layout (documented with the repack entry point) is, in words:
    tiles of 128 output rows in order; inside a tile, units of KB = max(128, G)
    input columns in order; a unit is its scale block then its code block.
    Scale block: for each group of the unit, for each 16-row slab, eight pairs
    (sw[row p], sw[row p+8]) for p = 0..7.  Code block: for each slab, for each
    pair of 16-wide k-steps, the 4-bit plane as 32 lanes x 2 words (step A then
    step B), then for 6-bit codes the 2-bit plane as 32 lanes x 1 word.  In a
    plane word of lane (g, t), A-register i's two elements sit at bits
    4i..4i+3 and 16+4i..16+4i+3 (low 4 bits of the code).  In the 2-bit plane
    word the top 2 bits of register i of step s (0 = A, 1 = B) sit at bits
    8s + 2*(i // 2) + 4*(i % 2) and 16 more than that.

    ``layout="codebook"`` (4-bit codes whose levels come from a codebook) is
    the same stream except inside a plane word: A-register i's two elements
    sit in byte i, the even k at bits 8i..8i+3 and the odd k at 8i+4..8i+7.

    ``layout="rows"`` (the row layout of the second main loop) keeps the
    tiles and units but orders each unit by rows: the scale block is
    [group][row]; the 4-bit plane holds, for each 32-wide k chunk c and each
    row, 4 little-endian words, word j holding the low 4 bits of the codes of
    k = 32c + 8j + i at bits 4i; for 6-bit codes the 2-bit plane follows,
    for each chunk and row 2 words, word h holding the top 2 bits of the codes
    of words 2h and 2h+1 of that row and chunk, code i at bit TOP2_POS[i]
    (plus 2 for word 2h+1).
    """
    if layout == "rows":
        return _unpack_stream_rows(fmt, N, K, G, buf)
    assert layout in ("plain", "codebook")
    assert layout == "plain" or fmt == "w4a8", "only 4-bit codes have the codebook layout"
    b = BITS[fmt]
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    assert N % 16 == 0 and K % 32 == 0 and K % G == 0
    KB = stream_kb(G)
    ROW, KIP = _slab_pair_index()
    reg = np.arange(4)[None, None, :, None]
    elem = np.arange(2)[None, None, None, :]
    step = np.arange(2)[None, :, None, None]
    nib_shift = (16 * elem + 4 * reg).astype(np.uint32)                 # [1,1,4,2]
    if layout == "codebook":
        nib_shift = (8 * reg + 4 * elem).astype(np.uint32)
    hi_shift = (8 * step + 16 * elem + 2 * (reg // 2) + 4 * (reg % 2)).astype(np.uint32)  # [1,2,4,2]
    codes = np.full((N, K), -1, dtype=np.int64)
    sw = np.full((N, K // G), np.nan, dtype=np.float32)
    pos = 0
    for t0 in range(0, N, STREAM_TN):
        R = min(STREAM_TN, N - t0)
        S = R // 16
        for k0 in range(0, K, KB):
            W = min(KB, K - k0)
            ng, P = W // G, W // 32
            # scale block: [group][slab][p][row p, row p+8]
            f = np.frombuffer(buf[pos:pos + 4 * R * ng].tobytes(), dtype="<f4").reshape(ng, S, 8, 2)
            pos += 4 * R * ng
            sw[t0:t0 + R, k0 // G:k0 // G + ng] = f.transpose(1, 3, 2, 0).reshape(R, ng)
            # code block: [slab][k-step pair][4-bit plane 32x2 words (+ 2-bit plane 32 words)]
            per = 256 + (128 if b == 6 else 0)
            blk = buf[pos:pos + S * P * per].reshape(S, P, per)
            pos += S * P * per
            nib = np.frombuffer(blk[:, :, :256].tobytes(), dtype="<u4").reshape(S, P, 32, 2, 1, 1)
            val = (nib >> nib_shift) & 0xF                                  # [S,P,32,2,4,2]
            if b == 6:
                hi = np.frombuffer(blk[:, :, 256:].tobytes(), dtype="<u4").reshape(S, P, 32, 1, 1, 1)
                val = val | (((hi >> hi_shift) & 0x3) << 4)
            tile = np.empty((S, 16, P, 32), dtype=np.int64)
            tile[:, ROW, :, KIP] = val.transpose(2, 3, 4, 5, 0, 1).astype(np.int64)
            codes[t0:t0 + R, k0:k0 + W] = tile.reshape(R, W)
    assert pos == file_bytes(fmt, N, K, G), (pos, file_bytes(fmt, N, K, G))
    assert codes.min() >= 0, "stream does not cover every (n, k)"
    return codes, sw


# Bit of the top 2 bits of code i (of a 4-bit plane word) in the row layout's
# 2-bit plane word, for the first word of the pair (the second is 2 bits up).
TOP2_POS = (4, 8, 0, 12, 20, 24, 16, 28)


def _unpack_stream_rows(fmt: str, N: int, K: int, G: int, buf) -> tuple[np.ndarray, np.ndarray]:
    """The row layout (see ``unpack_stream``), read unit by unit."""
    b = BITS[fmt]
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    assert N % 16 == 0 and K % 32 == 0 and K % G == 0 and G >= 32
    KB = stream_kb(G)
    i = np.arange(8)
    j = np.arange(4)
    top_shift = (np.array(TOP2_POS)[None, :] + 2 * (j[:, None] % 2)).astype(np.uint32)   # [word j, code i]
    codes = np.full((N, K), -1, dtype=np.int64)
    sw = np.full((N, K // G), np.nan, dtype=np.float32)
    pos = 0
    for t0 in range(0, N, STREAM_TN):
        R = min(STREAM_TN, N - t0)
        for k0 in range(0, K, KB):
            W = min(KB, K - k0)
            ng, C = W // G, W // 32
            f = np.frombuffer(buf[pos:pos + 4 * R * ng].tobytes(), dtype="<f4").reshape(ng, R)
            pos += 4 * R * ng
            sw[t0:t0 + R, k0 // G:k0 // G + ng] = f.T
            words = np.frombuffer(buf[pos:pos + R * W // 2].tobytes(), dtype="<u4").reshape(C, R, 4)
            pos += R * W // 2
            val = (words[..., None] >> (4 * i).astype(np.uint32)) & 0xF                 # [chunk, row, word, code]
            if b == 6:
                top = np.frombuffer(buf[pos:pos + R * W // 4].tobytes(), dtype="<u4").reshape(C, R, 2)
                pos += R * W // 4
                val = val | (((top[:, :, j // 2][..., None] >> top_shift) & 0x3) << 4)
            codes[t0:t0 + R, k0:k0 + W] = val.transpose(1, 0, 2, 3).reshape(R, W).astype(np.int64)
    assert pos == file_bytes(fmt, N, K, G), (pos, file_bytes(fmt, N, K, G))
    assert codes.min() >= 0, "stream does not cover every (n, k)"
    return codes, sw
