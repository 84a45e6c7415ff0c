"""CPU tier: the shared-memory layout of the tcgen05 projection kernel
(gemv_umma.cuh) checked access by access, with no GPU.

For every token count the kernel takes (16 to 64), feature counts from 32
to 6720 (small and ragged ones, the decode and Qwen3 widths, and those at
the edges of what fits), with and without the residual, and every cluster
size that fits, the areas are laid out as the kernel lays them out. The
accesses the kernel makes to them are then walked:
- the y, r and A atoms of each rank's K slice;
- the 16-byte chunks the norm reads and writes;
- the receive slots of each 4-token group;
- w's chunks, the mbarriers, the words, the partial sums and rstd.

Each access must stay inside its own area, and the areas may not overlap,
except the overlay the kernel relies on: receive over r (read before any
peer stores into it).
"""
import pytest

from tests.test_gemv_gpu import umma_layout_bytes

SMEM = 227 * 1024


def layout(T, H, KS, res):
    """Offsets as gemv_umma_layout computes them (bytes from the 1024-byte
    aligned base)."""
    na = (H + 63) // 64
    apc = (na + KS - 1) // KS
    rs = ((T // 4 + KS - 1) // KS) | 1
    atom = T * 128
    ybytes = apc * atom
    rbytes = ybytes if res else 0
    abytes = apc * 16384
    xchg = KS * 128 * rs * 16
    L = {"apc": apc, "rs": rs, "na": na, "atom": atom}
    L["y"] = (0, ybytes)
    L["r"] = (ybytes, ybytes + rbytes)
    L["a"] = (ybytes + rbytes, ybytes + rbytes + abytes)
    end = L["a"][1]
    if rbytes >= xchg:
        L["recv"] = (L["r"][0], L["r"][0] + xchg)
    else:
        L["recv"] = (end, end + xchg)
        end += xchg
    L["w"] = (end, end + apc * 128)
    bar = L["w"][1]
    L["bar"] = (bar, bar + 8 * (apc + 3))
    L["slots"] = (L["bar"][1], L["bar"][1] + 16)
    L["part"] = (L["slots"][1], L["slots"][1] + 4 * T)
    L["rsv"] = (L["part"][1], L["part"][1] + 4 * T)
    L["total"] = L["rsv"][1] + 1023
    return L


def inside(area, off, size):
    lo, hi = area
    return lo <= off and off + size <= hi


# feature counts: small and ragged ones, the decode and Qwen3 widths, and
# those at the edges of what fits
HS = (32, 64, 96, 128, 160, 896, 1024, 1664, 1696, 2048, 2272, 2304, 3072, 3136,
      3424, 3584, 3616, 4096, 4608, 4640, 5120, 5632, 5664, 6720)


def configs():
    for T in (16, 32, 48, 64):
        for res in (False, True):
            for H in HS:
                na = (H + 63) // 64
                for KS in range(1, min(8, na) + 1):
                    if umma_layout_bytes(T, H, KS, res) <= SMEM:
                        yield T, H, KS, res


def test_layout_matches_the_size_model():
    for T, H, KS, res in configs():
        assert layout(T, H, KS, res)["total"] == umma_layout_bytes(T, H, KS, res)


def test_every_access_stays_in_its_area():
    n = 0
    for T, H, KS, res in configs():
        L = layout(T, H, KS, res)
        na, apc, atom, rs = L["na"], L["apc"], L["atom"], L["rs"]
        NP = H // 8
        # areas disjoint but for the two overlays
        names = ["y", "r", "a", "w", "bar", "slots", "part", "rsv"]
        if L["recv"][0] != L["r"][0]:
            names.append("recv")
        spans = sorted(L[k] for k in names if L[k][1] > L[k][0])
        for (lo1, hi1), (lo2, hi2) in zip(spans, spans[1:]):
            assert hi1 <= lo2, (T, H, KS, res)
        if L["recv"][0] == L["r"][0]:
            assert L["recv"][1] <= L["r"][1]
        assert L["total"] <= SMEM
        G4 = T // 4
        for rank in range(KS):
            a0 = rank * na // KS
            nat = (rank + 1) * na // KS - a0
            assert 1 <= nat <= apc <= 32
            for i in range(nat):
                # A atom, x/y atom, r atom (tensor copies and MMA operands)
                assert inside(L["a"], L["a"][0] + i * 16384, 16384)
                assert inside(L["y"], L["y"][0] + i * atom, atom)
                if res:
                    assert inside(L["r"], L["r"][0] + i * atom, atom)
                # the norm's chunks of the first rows, a swizzle period on
                # and the last row
                for row in sorted({0, 1, 7, 8, 9, T - 1}):
                    for c8 in range(8):
                        if (a0 + i) * 8 + c8 >= NP:
                            continue
                        off = i * atom + row * 128 + ((c8 ^ (row & 7)) << 4)
                        assert inside(L["y"], L["y"][0] + off, 16)
                        if res:
                            assert inside(L["r"], L["r"][0] + off, 16)
                        assert inside(L["w"], L["w"][0] + (i * 8 + c8) * 16, 16)
            # exchange: every group's slot at its owner, from every rank
            own = (G4 - 1 - rank) // KS + 1 if G4 > rank else 0
            for g in range(G4):
                owner, slot = g % KS, g // KS
                assert slot < rs
                for fl in (0, 127):
                    off = ((rank * 128 + fl) * rs + slot) * 16
                    assert inside((0, L["recv"][1] - L["recv"][0]), off, 16)
            for slot in range(own):
                assert slot * KS + rank < G4
            # a rank's block of the receive area, 16-byte stores
            block = 128 * rs * 16
            assert (rank + 1) * block <= L["recv"][1] - L["recv"][0]
            assert block % 16 == 0
        n += 1
    assert n > 300
