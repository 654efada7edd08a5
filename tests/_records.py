"""The per-tile records of the two-pass forward, restated from their
definition (integer work, compared exactly with the list pass on the GPU)."""

import numpy as np

TILE, MAXREC = 16, 7


def records_ref(idx, N, bs):
    """[B, G, tiles, 8] int32: count, then up to 7 ids -- the blocks listed by
    every query of the tile, in the order the tile's first query lists them,
    whose first key is <= the first query's position and whose keys all lie
    below min(M, N)."""
    B, M, G, T = idx.shape
    nblk = -(-N // bs)
    ntiles = -(-M // TILE)
    out = np.full((B, G, ntiles, 8), -1, np.int32)
    for b in range(B):
        for g in range(G):
            for t in range(ntiles):
                m0 = t * TILE
                rows = idx[b, m0:min(M, m0 + TILE), g]
                sets = [set(r.tolist()) for r in rows]
                lim = min(M, N)
                ids = []
                for e in rows[0].tolist():
                    if len(ids) == MAXREC:
                        break
                    if 0 <= e < nblk and e * bs <= m0 and (e + 1) * bs <= lim and \
                            e not in ids and \
                            all(e in s for s in sets):
                        ids.append(e)
                out[b, g, t, 0] = len(ids)
                out[b, g, t, 1:1 + len(ids)] = ids
    return out
