"""Exhaustive bit-exact check of the fused-quantization append: every finite
bf16 value is encoded under a set of group maxima (anchors), on the GPU
through nk_paged_kv_append and in the oracle codec, and the bytes compared.

Each quantization group starts with its anchor (the group's amax) followed by
bf16 values of magnitude <= anchor, so every quotient x / s the hardware
conversions see lies in the codec's working range, including ties, -0.0,
subnormal fp16 scales and saturated E4M3 scales."""

import numpy as np
import pytest
import torch

from oracle import codec, formats as F
from paged_kv_cache_append_gb300 import nk

pytestmark = pytest.mark.gpu

# the last three put amax / 127 and amax / 448 past the largest finite
# binary16, where the INT8-G64 and FP8-row scales saturate at 65504
ANCHORS = [1.0, 1.0078125, 3.140625, 448.0, 449.0, 127.0, 6.0, 2688.0, 1.0e-3, 6.0e-5,
           2.0 ** -20, 2.5e4, 1.0e6, 0.75, 254 * 32768.0, 2.0 ** 26, 3.0e38]
GROUP = {"int8_g64": 64, "fp8_row": 256, "nvfp4_g16": 16}


def _all_finite_bf16():
    bits = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    x = F.bf16_bits_to_f64(bits)
    return bits[np.isfinite(x)], x[np.isfinite(x)]


def _rows_for(kind, seed):
    bits, x = _all_finite_bf16()
    g = GROUP[kind]
    rng = np.random.default_rng(seed)
    rows = []
    for A in ANCHORS:
        a_bits = F.f64_to_bf16_bits(np.array([A]))[0]
        a = F.bf16_bits_to_f64(np.array([a_bits]))[0]
        sel = bits[np.abs(x) <= a]
        sel = sel[rng.permutation(sel.size)]
        per = g - 1
        n = -(-sel.size // per)
        grp = np.full((n, g), a_bits, dtype=np.uint16)
        flat = np.concatenate([sel, np.zeros(n * per - sel.size, np.uint16)])
        grp[:, 1:] = flat.reshape(n, per)
        # alternate the anchor's sign and position inside the group
        pos = rng.integers(0, g, n)
        grp[np.arange(n), 0], grp[np.arange(n), pos] = grp[np.arange(n), pos], grp[np.arange(n), 0]
        flip = rng.random(n) < 0.5
        grp[flip, pos[flip]] ^= 0x8000
        rows.append(grp.reshape(-1))
    v = np.concatenate(rows)
    v = np.concatenate([v, np.zeros((-v.size) % 256, np.uint16)])
    return v.reshape(-1, 256)              # [tokens, D=256]


@pytest.mark.parametrize("profile,kind", [("int8_g64", "int8_g64"), ("fp8_row", "fp8_row"),
                                          ("nvfp4_g16", "nvfp4_g16")])
def test_codec_exhaustive_bf16(profile, kind):
    kb = _rows_for(kind, 1)
    vb = _rows_for(kind, 2)[: kb.shape[0]]
    if vb.shape[0] < kb.shape[0]:
        vb = np.concatenate([vb, kb[vb.shape[0]:]])
    T = kb.shape[0]
    S = -(-T // 64) * 64
    pool = nk.Pool(profile, 1, 1, 256, S, 1, S // 64)
    L = S // 64
    table = np.random.default_rng(3).permutation(L).astype(np.int32)[None, :]
    dev = "cuda"
    k = torch.from_numpy(kb.view(np.int16).copy()).view(torch.bfloat16).reshape(1, T, 1, 256)
    v = torch.from_numpy(vb.view(np.int16).copy()).view(torch.bfloat16).reshape(1, T, 1, 256)
    pool.append(0, torch.from_numpy(table).to(dev), torch.zeros(1, dtype=torch.int32, device=dev),
                torch.zeros(1, dtype=torch.int32, device=dev), k.to(dev), v.to(dev))
    torch.cuda.synchronize()
    want = codec.encode_kv(profile, kb[:, None, :], vb[:, None, :])
    pos = np.arange(T)
    g = table[0, pos // 64]
    for i, name in enumerate(["k", "v", "k_scale", "v_scale"]):
        rb = pool.row_bytes[i]
        plane = pool.planes[0][i].cpu().numpy().reshape(L, 1, 64, rb)
        got = plane[g, 0, pos % 64]
        exp = want[name][:, 0]
        if not np.array_equal(got, exp):
            bad = np.argwhere(got != exp)
            t0, c0 = bad[0]
            raise AssertionError(
                f"{profile} plane {name}: {len(bad)} bytes differ; first token {t0} byte {c0}: "
                f"gpu {got[t0, c0]:#04x} oracle {exp[t0, c0]:#04x}; "
                f"inputs k[{t0}, :8] = {[hex(x) for x in kb[t0, :8]]}")
