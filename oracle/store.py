"""Byte image of a typed growing KV pool (test infrastructure only).

Follows the "Paged KV cache" maintainer design page of the NInfer engine:

* every plane of every layer is a separate byte array with closed strides in
  the page-major order [X, P, H, N_physical] (physical layout section);
* one page-group id g selects slice g in all planes of all layers, so the
  code and scale planes of a token share g (page grouping section);
* append writes the codes and scales of token position ``pos`` of compact row
  b at (g, o) = (block_tables[table_rows[b]][pos >> 6], pos & 63) (consumer
  view section, translation);
* gather reads logical positions 0..F-1 of one table row back and
  dequantizes them (a consumer reads the pages in place; the gather here is
  only the oracle's way of forming the logical sequence);
* ``copy_columns`` is the partial-tail copy-on-write of the Fork worked
  example: the committed columns of the source tail page are copied into a
  private destination page for every plane and layer, full pages are shared;
* ``pack_pages`` / ``unpack_pages`` form the host replica of the host replica
  section: pages in logical order without device ids, each packed page holding
  the whole grouped payload (for each layer, each plane: every (h, o) row of
  that page group, in the plane's own (h, o) order).

Parity pins: bit-exact planes against the CUDA append; invariance of gathered
values under a random permutation of physical ids; the F = 1000 Fork example.
"""

from __future__ import annotations

import numpy as np

from . import codec, layout


class PoolImage:
    """All planes of a pool as zero-initialised host byte arrays."""

    def __init__(self, profile: str, num_layers: int, H: int, D: int, M: int,
                 order: str = "page_major"):
        self.profile, self.num_layers, self.H, self.D, self.M = profile, num_layers, H, D, M
        self.order = order
        self.schema = layout.plane_schema(profile, D)
        self.planes = [[np.zeros(layout.plane_bytes(p, H, M), dtype=np.uint8)
                        for p in self.schema] for _ in range(num_layers)]

    # -- addressing ------------------------------------------------------
    def _row_slice(self, pi: int, o: int, h: int, g: int) -> slice:
        p = self.schema[pi]
        a = layout.address(p, self.H, self.M, 0, o, h, g, self.order)
        return slice(a, a + p.row_bytes)

    # -- write -----------------------------------------------------------
    def write_token(self, layer: int, g: int, o: int, k_bits: np.ndarray, v_bits: np.ndarray) -> None:
        """Encode and store one token (all heads): k_bits, v_bits uint16 [H, D]."""
        rows = codec.encode_kv(self.profile, k_bits, v_bits)
        for pi, p in enumerate(self.schema):
            for h in range(self.H):
                self.planes[layer][pi][self._row_slice(pi, o, h, g)] = rows[p.name][h]

    def append(self, layer: int, block_tables: np.ndarray, table_rows: np.ndarray,
               write_pos: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray,
               counts: np.ndarray | None = None) -> None:
        """Append T tokens per compact row b at positions write_pos[b] + t.

        block_tables int32 [C, L]; table_rows int32 [B]; write_pos int32 [B];
        k_bits / v_bits uint16 [B, T, H, D]; counts[b] <= T limits the tokens
        written for row b (all T when None).
        """
        B, T = k_bits.shape[:2]
        for b in range(B):
            row = block_tables[table_rows[b]]
            n = T if counts is None else int(counts[b])
            for t in range(n):
                g, o = layout.translate(int(write_pos[b]) + t, row)
                self.write_token(layer, g, o, k_bits[b, t], v_bits[b, t])

    # -- read ------------------------------------------------------------
    def read_rows(self, layer: int, table_row: np.ndarray, F: int) -> dict[str, np.ndarray]:
        """Plane bytes of logical positions [0, F) -> {name: uint8 [F, H, row_bytes]}."""
        out = {p.name: np.zeros((F, self.H, p.row_bytes), dtype=np.uint8) for p in self.schema}
        for pos in range(F):
            g, o = layout.translate(pos, table_row)
            for pi, p in enumerate(self.schema):
                for h in range(self.H):
                    out[p.name][pos, h] = self.planes[layer][pi][self._row_slice(pi, o, h, g)]
        return out

    def gather(self, layer: int, table_row: np.ndarray, F: int) -> tuple[np.ndarray, np.ndarray]:
        """Dequantized (K, V) float64 [F, H, D] of logical positions [0, F)."""
        return codec.decode_kv(self.profile, self.read_rows(layer, table_row, F))

    # -- copy-on-write ---------------------------------------------------
    def copy_columns(self, g_src: int, g_dst: int, ncols: int) -> None:
        """Copy columns [0, ncols) of page group g_src into g_dst, every plane
        and layer (private partial tail of a Fork)."""
        for layer in range(self.num_layers):
            for pi in range(len(self.schema)):
                for h in range(self.H):
                    for o in range(ncols):
                        self.planes[layer][pi][self._row_slice(pi, o, h, g_dst)] = \
                            self.planes[layer][pi][self._row_slice(pi, o, h, g_src)]

    # -- host replica --------------------------------------------------------
    def packed_page_bytes(self) -> int:
        return self.num_layers * sum(p.row_bytes * layout.P * self.H for p in self.schema)

    def pack_pages(self, page_ids) -> np.ndarray:
        """Host replica of pages page_ids (logical order): uint8 [n, page bytes]."""
        out = []
        for g in page_ids:
            parts = []
            for layer in range(self.num_layers):
                for pi in range(len(self.schema)):
                    for h in range(self.H):
                        for o in range(layout.P):
                            parts.append(self.planes[layer][pi][self._row_slice(pi, o, h, int(g))])
            out.append(np.concatenate(parts))
        return np.stack(out) if out else np.zeros((0, self.packed_page_bytes()), np.uint8)

    def unpack_pages(self, page_ids, packed: np.ndarray) -> None:
        """Writes a host replica back into page groups page_ids."""
        for i, g in enumerate(page_ids):
            at = 0
            for layer in range(self.num_layers):
                for pi, p in enumerate(self.schema):
                    for h in range(self.H):
                        for o in range(layout.P):
                            self.planes[layer][pi][self._row_slice(pi, o, h, int(g))] = \
                                packed[i, at:at + p.row_bytes]
                            at += p.row_bytes
