"""Pool geometry of a typed growing KV pool (test infrastructure only).

Follows the "Paged KV cache" maintainer design page of the NInfer engine:

* page size P = 64 tokens (granularity table; "P=64" rationale paragraph);
* capacity bounds L = ceil(S/P), M_min = max(L, C), M_max = C*L and the
  explicit policy M = ceil(K_main/P) with K_main >= S (capacity section);
* closed plane orders: page-major [X, P, H, N_physical] for Main/MTP pools and
  head-major [X, P, N_physical, H] for the draft pool, innermost first, with
  byte address  base + d*nb0 + o*nb1 + h*nb2 + g*nb3  (page-major) and
  base + d*nb0 + o*nb1 + g*nb2 + h*nb3 (head-major) (physical layout section);
* plane extents X: code plane X = D, INT8-G64 scale X = D/64, FP8-row scale
  X = 1, NVFP4 packed codes X = D/2 and scales X = D/16 (same section);
* the per-token/head byte table for D = 256 (BF16 1024 B, INT8-G64 528 B,
  FP8-E4M3FN-row256 516 B, NVFP4-G16 288 B, K8V4 402 B) and
  PageBytes = sum over planes of bytes/token * P;
* translation: logical block = pos >> 6, page offset = pos & 63,
  physical page = block_table[logical block]; batched consumers first pick
  the table row with table_rows[b] (consumer view section).

Reading of the pages taken here (stated, not printed there): a profile's planes
are ordered [K code, V code, K scale, V scale]; scale planes of INT8-G64 and
FP8-row hold IEEE binary16 (2 bytes, matching the byte table); NVFP4 scales
are E4M3FN bytes.

* speculative backends (pool geometry and trim paragraphs): the MTP pool of a
  draft window K holds M + C * ceil((K - 1) / P) pages, the lead of each
  active row over Main in one speculative round; a row keeps
  ceil(max(committed, provisional) / P) logical pages mapped and may release
  the trailing ones, the last partial page included in what it keeps.

Pinned by: the byte table and the Fork/COW worked example printed on the page
(tests/golden), the closed-form M bounds, hand-computed addresses, and brute
force over frontier offsets for the speculative page counts.
"""

from __future__ import annotations

from dataclasses import dataclass

P = 64
PROFILES = ("bf16", "int8_g64", "fp8_row", "nvfp4_g16", "k8v4")
PROFILE_ID = {name: i for i, name in enumerate(PROFILES)}


@dataclass(frozen=True)
class Plane:
    name: str        # "k", "v", "k_scale", "v_scale"
    elem_bytes: int  # bytes per element of the plane
    X: int           # leading extent (elements per token per head)

    @property
    def row_bytes(self) -> int:
        return self.X * self.elem_bytes


def plane_schema(profile: str, D: int) -> list[Plane]:
    """Planes of one layer for a KV profile, in plane-ordinal order."""
    if profile == "bf16":
        return [Plane("k", 2, D), Plane("v", 2, D)]
    if profile == "int8_g64":
        return [Plane("k", 1, D), Plane("v", 1, D),
                Plane("k_scale", 2, D // 64), Plane("v_scale", 2, D // 64)]
    if profile == "fp8_row":
        return [Plane("k", 1, D), Plane("v", 1, D),
                Plane("k_scale", 2, 1), Plane("v_scale", 2, 1)]
    if profile == "nvfp4_g16":
        return [Plane("k", 1, D // 2), Plane("v", 1, D // 2),
                Plane("k_scale", 1, D // 16), Plane("v_scale", 1, D // 16)]
    if profile == "k8v4":
        return [Plane("k", 1, D), Plane("v", 1, D // 2),
                Plane("k_scale", 2, 1), Plane("v_scale", 1, D // 16)]
    raise ValueError(f"unknown profile {profile!r}")


def bytes_per_token_head(profile: str, D: int) -> int:
    return sum(p.row_bytes for p in plane_schema(profile, D))


def page_bytes(profile: str, D: int, H: int, num_layers: int = 1) -> int:
    """PageBytes = sum over planes of bytes per token * P (all heads, layers)."""
    return bytes_per_token_head(profile, D) * H * P * num_layers


def strides(plane: Plane, H: int, M: int, order: str = "page_major") -> tuple[int, int, int, int]:
    """Closed byte strides (nb0, nb1, nb2, nb3), innermost first."""
    nb0 = plane.elem_bytes
    nb1 = plane.X * nb0
    nb2_inner = P * nb1
    if order == "page_major":       # [X, P, H, N]
        return nb0, nb1, nb2_inner, H * nb2_inner
    if order == "head_major":       # [X, P, N, H]
        return nb0, nb1, nb2_inner, M * nb2_inner
    raise ValueError(order)


def address(plane: Plane, H: int, M: int, d: int, o: int, h: int, g: int,
            order: str = "page_major") -> int:
    """Byte offset of element (d, o, h, g) from the plane base."""
    nb0, nb1, nb2, nb3 = strides(plane, H, M, order)
    if order == "page_major":
        return d * nb0 + o * nb1 + h * nb2 + g * nb3
    return d * nb0 + o * nb1 + g * nb2 + h * nb3


def plane_bytes(plane: Plane, H: int, M: int) -> int:
    return plane.row_bytes * P * H * M


def logical_pages(S: int) -> int:
    """L = ceil(S / P)."""
    return -(-S // P)


def m_bounds(S: int, C: int) -> tuple[int, int]:
    """(M_min, M_max) = (max(L, C), C * L)."""
    L = logical_pages(S)
    return max(L, C), C * L


def explicit_capacity(K_main: int, S: int, C: int) -> int:
    """Explicit kv_capacity policy: M = ceil(K_main / P); requires K_main >= S
    and M in [M_min, M_max]; raises ValueError otherwise."""
    if K_main < S:
        raise ValueError("K_main must be >= max_context")
    M = -(-K_main // P)
    lo, hi = m_bounds(S, C)
    if not lo <= M <= hi:
        raise ValueError(f"M={M} outside [{lo}, {hi}]")
    return M


def translate(pos: int, table_row) -> tuple[int, int]:
    """(physical page g, page offset o) of logical position ``pos``."""
    return int(table_row[pos >> 6]), pos & 63


def fork_split(F: int) -> tuple[int, int]:
    """Fork of a frontier F: (number of full immutable pages shared,
    committed columns of the partial tail copied to a private page)."""
    return F // P, F % P


def mtp_pages(M: int, C: int, K: int) -> int:
    """Physical pages of the MTP backend pool for draft window K (>= 1):
    M + C * ceil((K - 1) / P)."""
    if K < 1:
        raise ValueError("draft window must be >= 1")
    return M + C * (-(-(K - 1) // P))


def pages_needed(committed: int, provisional: int) -> int:
    """Logical pages a row keeps mapped: ceil(max(committed, provisional) / P)."""
    if committed < 0 or provisional < 0:
        raise ValueError("frontiers must be >= 0")
    return -(-max(committed, provisional) // P)
