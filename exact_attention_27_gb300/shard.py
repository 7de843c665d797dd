"""Data-parallel partition of the attention work (no exchange between parts).

A unit of work is one (batch, key/value head) pair together with the G query
heads that read that K/V head (G = H_q / H_kv).  Units are independent in the
forward and the backward pass; a unit must stay whole on one device so that
dK and dV need no cross-device reduction.  With the [B][H][N][d] layout a
contiguous range of units is contiguous memory in every tensor, and is itself
a valid call of the library with B' = number of units, H_q' = G, H_kv' = 1.

These helpers only compute ranges and tensor views; they launch nothing.
"""


def unit_count(B, Hq, Hkv):
    if Hq % Hkv:
        raise ValueError("H_q must be a multiple of H_kv")
    return B * Hkv


def unit_range(rank, world, n_units):
    """Contiguous [start, stop) of units for `rank` of `world` (sizes differ by at most 1)."""
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    base, rem = divmod(n_units, world)
    start = rank * base + min(rank, rem)
    return start, start + base + (1 if rank < rem else 0)


def unit_view(t, heads_per_unit, start, stop):
    """Rows [start, stop) of t seen as [units, heads_per_unit, ...].

    t is [B, H, ...] contiguous with H a multiple of heads_per_unit; the view
    shares t's storage and is contiguous."""
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    B, H = t.shape[0], t.shape[1]
    if H % heads_per_unit:
        raise ValueError("head count is not a multiple of heads_per_unit")
    return t.reshape(B * H // heads_per_unit, heads_per_unit, *t.shape[2:])[start:stop]


def shard(tensors, Hq, Hkv, rank, world):
    """Views of one rank's units.

    tensors: dict of name -> tensor; names starting with "q", "o", "lse", "dq",
    "do" or "D" carry H_q heads, "k", "v", "dk", "dv" carry H_kv heads.
    Returns (views, (B', H_q', H_kv')) for the library call on the shard."""
    G = Hq // Hkv
    any_t = next(iter(tensors.values()))
    n_units = unit_count(any_t.shape[0], Hq, Hkv)
    start, stop = unit_range(rank, world, n_units)
    out = {}
    for name, t in tensors.items():
        per_unit = G if t.shape[1] == Hq else 1
        if t.shape[1] not in (Hq, Hkv):
            raise ValueError(f"{name}: head dimension {t.shape[1]} is neither H_q nor H_kv")
        if Hq == Hkv:
            per_unit = 1
        out[name] = unit_view(t, per_unit, start, stop)
    return out, (stop - start, G, 1)
