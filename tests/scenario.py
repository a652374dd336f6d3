"""Builds the same paged-KV state on the GPU (through libnk) and in the oracle
(through oracle.store) from one seeded workload, for the parity tests.

Both sides start from the same bf16 inputs drawn by
paged_kv_cache_append_gb300.workloads; neither reads the other's results.
"""

from __future__ import annotations

import numpy as np
import torch

from oracle import attention as OA
from oracle import codec as OC
from oracle import formats as OF
from oracle.store import PoolImage
from paged_kv_cache_append_gb300 import nk
from paged_kv_cache_append_gb300.workloads import Workload, bf16_to_bits

P = 64


def _pad_rows(chunks, H, D):
    """List of [n_b, H, D] bf16 tensors -> ([B, Tmax, H, D], counts)."""
    Tm = max(1, max(c.shape[0] for c in chunks))
    out = torch.zeros((len(chunks), Tm, H, D), dtype=torch.bfloat16)
    for i, c in enumerate(chunks):
        out[i, :c.shape[0]] = c
    return out, np.array([c.shape[0] for c in chunks], np.int32)


class Scenario:
    """Context fill of every table row (with an optional shared prefix and
    copy-on-write tail), one decode step per layer: append T tokens per decode
    row, then attend."""

    def __init__(self, w: Workload, layers=(0,), device="cuda", oracle=True, check_bounds=False,
                 order="page_major"):
        self.w, self.layers, self.device, self.with_oracle = w, list(layers), device, oracle
        self.gpu = nk.Pool(w.profile, w.num_layers, w.Hkv, w.D, w.S, w.C, w.M, device=device,
                           check_bounds=check_bounds, order=order)
        self.orc = PoolImage(w.profile, w.num_layers, w.Hkv, w.D, w.M, order=order) if oracle else None
        self.tables_d = torch.from_numpy(w.tables).to(device)
        self._fill()

    # -- context --------------------------------------------------------
    def row_context(self):
        """Tokens each table row holds before the step: decode rows hold
        context[b]; prefill rows hold their prefix."""
        n = np.zeros(self.w.C, np.int64)
        n[self.w.table_rows] = self.w.context
        if len(self.w.prefill_rows):
            n[self.w.prefill_rows] = self.w.prefix_len
        return n

    def _fill(self):
        w = self.w
        ctx = self.row_context()
        sh = w.shared_len
        full, tail = sh // P, sh % P
        vals = {layer: [w.context_kv(layer, r, int(ctx[r])) for r in range(w.C)] for layer in self.layers}
        if sh:
            # row 0 writes the shared prefix, the other rows share its full
            # pages and get a private copy of its partial tail page (Fork)
            for layer in self.layers:
                k0, v0 = vals[layer][0]
                self._append_rows(layer, [0], [0], [k0[:sh]], [v0[:sh]])
            if tail:
                for r in range(1, w.C):
                    src, dst = int(w.tables[0, full]), int(w.tables[r, full])
                    self.gpu.copy_columns(src, dst, tail)
                    if self.orc is not None:
                        self.orc.copy_columns(src, dst, tail)
        for layer in self.layers:
            rows = list(range(w.C))
            self._append_rows(layer, rows, [sh] * w.C, [vals[layer][r][0][sh:] for r in rows],
                              [vals[layer][r][1][sh:] for r in rows])
        torch.cuda.synchronize()

    def _append_rows(self, layer, rows, start, ks, vs):
        w = self.w
        live = [i for i in range(len(rows)) if ks[i].shape[0] > 0]
        if not live:
            return
        rows = [rows[i] for i in live]
        start = [start[i] for i in live]
        k, counts = _pad_rows([ks[i] for i in live], w.Hkv, w.D)
        v, _ = _pad_rows([vs[i] for i in live], w.Hkv, w.D)
        dev = self.device
        tr = torch.tensor(rows, dtype=torch.int32, device=dev)
        wp = torch.tensor(start, dtype=torch.int32, device=dev)
        ct = torch.from_numpy(counts).to(dev)
        self.gpu.append(layer, self.tables_d, tr, wp, k.to(dev).contiguous(), v.to(dev).contiguous(),
                        counts=ct)
        if self.orc is not None:
            self.orc.append(layer, self.w.tables, np.array(rows), np.array(start),
                            bf16_to_bits(k), bf16_to_bits(v), counts=counts)

    # -- decode step ---------------------------------------------------------
    def step(self, layer, out=None, lse=None, fused=False):
        """Appends the step tokens of the decode rows and runs the GPU decode
        (fused=True: both in one nk_paged_append_decode_attention call).
        Returns (q, out, lse, frontiers) with q on the CPU."""
        w = self.w
        k, v = w.step_kv(layer)
        q = w.step_q(layer)
        dev = self.device
        tr = torch.from_numpy(w.table_rows).to(dev)
        wp = torch.from_numpy(w.context).to(dev)
        fr = torch.from_numpy(w.context + w.T).to(dev)
        if self.orc is not None:
            self.orc.append(layer, w.tables, w.table_rows, w.context, bf16_to_bits(k), bf16_to_bits(v))
        if fused:
            o, l = self.gpu.append_decode(layer, q.to(dev), k.to(dev), v.to(dev), self.tables_d, tr, fr,
                                          w.scale, out=out, lse=lse)
        else:
            self.gpu.append(layer, self.tables_d, tr, wp, k.to(dev), v.to(dev))
            o, l = self.gpu.decode(layer, q.to(dev), self.tables_d, tr, fr, w.scale, out=out, lse=lse)
        torch.cuda.synchronize()
        return q, o.cpu(), l.cpu(), w.context + w.T

    def oracle_decode(self, layer, q, frontiers):
        w = self.w
        qf = OF.bf16_bits_to_f64(bf16_to_bits(q))
        outs, lses = [], []
        for b in range(w.B):
            K, V = self.orc.gather(layer, w.tables[w.table_rows[b]], int(frontiers[b]))
            o, l = OA.decode(qf[b], K, V, int(frontiers[b]), w.scale)
            outs.append(o)
            lses.append(l)
        return np.stack(outs), np.stack(lses)

    def planes_equal(self, layer):
        """Bit-exact comparison of every plane of a layer (GPU vs oracle)."""
        bad = []
        for i, t in enumerate(self.gpu.planes[layer]):
            g = t.cpu().numpy()
            o = self.orc.planes[layer][i]
            if not np.array_equal(g, o):
                idx = np.flatnonzero(g != o)
                bad.append((i, idx.size, int(idx[0]), int(g[idx[0]]), int(o[idx[0]])))
        return bad


def oracle_row(w: Workload, layer: int, b: int):
    """Oracle (out [T, Hq, D], lse [T, Hq]) of decode row b after its step
    append, from the host inputs alone: encodes only that row's context and
    step tokens (rows that share a prefix read row 0's values there)."""
    r = int(w.table_rows[b])
    n = int(w.context[b])
    sh = w.shared_len
    kc, vc = w.context_kv(layer, r, n)
    if sh and r != 0:
        k0, v0 = w.context_kv(layer, 0, int(w.context[0]))
        kc = torch.cat([k0[:sh], kc[sh:]])
        vc = torch.cat([v0[:sh], vc[sh:]])
    ks, vs = w.step_kv(layer)
    kb = np.concatenate([bf16_to_bits(kc), bf16_to_bits(ks[b])], axis=0)
    vb = np.concatenate([bf16_to_bits(vc), bf16_to_bits(vs[b])], axis=0)
    K, V = OC.decode_kv(w.profile, OC.encode_kv(w.profile, kb, vb))
    q = OF.bf16_bits_to_f64(bf16_to_bits(w.step_q(layer)[b]))
    return OA.decode(q, K, V, n + w.T, w.scale)


def compare_attention(out, lse, ref_out, ref_lse, atol_out=2e-2, atol_lse=1e-3, strict=False,
                      ref_rounded=False, extra=None):
    """Checks the GPU output against the oracle.

    out: |gpu - oracle| <= 2e-2 + 2^-8 |oracle|, i.e. 2e-2 absolute beyond the
    rounding of the bf16 output itself (round to nearest moves a value of
    magnitude |o| by at most half an ulp, 2^-8 |o|, which alone exceeds 2e-2
    once |o| > 5, as with the x20 outliers).
    lse: |gpu - oracle| <= 1e-3 where finite; -inf exactly where the oracle
    has no key.  strict=True drops the ulp term (plain 2e-2 absolute).
    ref_rounded=True: the reference is itself a bf16 output (another GPU
    path), so each side's rounding contributes half an ulp: 2^-7 |ref|.
    extra: a further per-element allowance (same shape as ref_out), for a
    path whose own rounding has a bound of its own.
    Returns (max out excess, max lse error)."""
    o = out.float().numpy().astype(np.float64)
    l = lse.numpy().astype(np.float64)
    assert np.all(np.isfinite(o)), "non-finite output"
    ulp_term = 0.0 if strict else (2.0 ** -7 if ref_rounded else 2.0 ** -8)
    excess = np.abs(o - ref_out) - ulp_term * np.abs(ref_out)
    if extra is not None:
        excess = excess - extra
    err_o = float(np.max(excess)) if o.size else 0.0
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(l), fin), "lse finiteness differs"
    err_l = float(np.max(np.abs(l[fin] - ref_lse[fin]))) if fin.any() else 0.0
    raw = float(np.max(np.abs(o - ref_out))) if o.size else 0.0
    assert err_o <= atol_out and err_l <= atol_lse, \
        f"out excess {err_o} (raw max-abs {raw}), lse max-abs error {err_l}"
    return err_o, err_l
