"""View algebra (host side): a View is (shape, strides, offset, mask) and the
movement ops compose into a single View at zero cost (limn, "Three rules hold
it together": reshape, permute, expand, pad and shrink compose into one View
and lower to index arithmetic).  Element i reads base[offset + sum i_d *
strides_d] when mask_lo_d <= i_d < mask_hi_d for every d, else zero.
"""
from __future__ import annotations

from math import prod


class View:
    __slots__ = ("shape", "strides", "offset", "mask")

    def __init__(self, shape, strides=None, offset=0, mask=None):
        self.shape = tuple(int(s) for s in shape)
        if strides is None:
            strides = View.row_major(self.shape)
        self.strides = tuple(int(s) for s in strides)
        self.offset = int(offset)
        self.mask = None if mask is None else tuple((int(a), int(b)) for a, b in mask)
        if self.mask is not None and all(lo <= 0 and hi >= s for (lo, hi), s in zip(self.mask, self.shape)):
            self.mask = None

    @staticmethod
    def row_major(shape):
        st, s = [0] * len(shape), 1
        for d in range(len(shape) - 1, -1, -1):
            st[d] = s if shape[d] != 1 else 0
            s *= shape[d]
        return tuple(st)

    def __repr__(self):
        return "View(%s, %s, off=%d, mask=%s)" % (self.shape, self.strides, self.offset, self.mask)

    def key(self):
        return (self.shape, self.strides, self.offset, self.mask)

    def numel(self):
        return prod(self.shape)

    def contiguous(self):
        return self.mask is None and self.offset == 0 and all(
            s == 1 or st == r for s, st, r in zip(self.shape, self.strides, View.row_major(self.shape)))

    def _mask(self):
        return self.mask if self.mask is not None else tuple((0, s) for s in self.shape)

    # ---- movement ----------------------------------------------------------
    def permute(self, perm):
        perm = tuple(perm)
        assert sorted(perm) == list(range(len(self.shape))), perm
        m = None if self.mask is None else tuple(self.mask[p] for p in perm)
        return View([self.shape[p] for p in perm], [self.strides[p] for p in perm], self.offset, m)

    def expand(self, shape):
        shape = tuple(shape)
        assert len(shape) == len(self.shape)
        st = []
        for s, n, t in zip(self.shape, shape, self.strides):
            assert s == n or s == 1, (self.shape, shape)
            st.append(t if s == n else 0)
        m = None
        if self.mask is not None:
            # an expanded size-1 dim keeps its mask (in or out for every index)
            m = tuple((lo, hi) if s == n else ((0, n) if lo <= 0 < hi else (0, 0))
                      for (lo, hi), s, n in zip(self.mask, self.shape, shape))
        return View(shape, st, self.offset, m)

    def shrink(self, arg):
        arg = tuple((int(a), int(b)) for a, b in arg)
        off = self.offset + sum(a * t for (a, _), t in zip(arg, self.strides))
        m = None
        if self.mask is not None:
            m = tuple((max(lo - a, 0), max(min(hi - a, b - a), 0)) for (lo, hi), (a, b) in zip(self.mask, arg))
        return View([b - a for a, b in arg], self.strides, off, m)

    def pad(self, arg):
        arg = tuple((int(a), int(b)) for a, b in arg)
        if all(a == 0 and b == 0 for a, b in arg):
            return self
        mk = self._mask()
        m = tuple((lo + a, hi + a) for (lo, hi), (a, _) in zip(mk, arg))
        off = self.offset - sum(a * t for (a, _), t in zip(arg, self.strides))
        return View([s + a + b for s, (a, b) in zip(self.shape, arg)], self.strides, off, m)

    def reshape(self, shape):
        """The same cells in a new shape, or None when no strided View can
        express it (then the source must be copied first)."""
        shape = tuple(int(s) for s in shape)
        assert prod(shape) == prod(self.shape), (self.shape, shape)
        if shape == self.shape:
            return self
        if self.mask is not None:
            return None
        old = [(s, t) for s, t in zip(self.shape, self.strides) if s != 1]
        new_st = [0] * len(shape)
        nz = [i for i, s in enumerate(shape) if s != 1]
        i = j = 0
        while i < len(old) or j < len(nz):
            if i >= len(old) or j >= len(nz):
                return None
            # grow one group on each side until the products agree
            gi, gj = [i], [nz[j]]
            po, pn = old[i][0], shape[nz[j]]
            i += 1
            j += 1
            while po != pn:
                if po < pn:
                    if i >= len(old):
                        return None
                    gi.append(i)
                    po *= old[i][0]
                    i += 1
                else:
                    if j >= len(nz):
                        return None
                    gj.append(nz[j])
                    pn *= shape[nz[j]]
                    j += 1
            # the old dims of the group must be one strided run
            for a, b in zip(gi, gi[1:]):
                if old[a][1] != old[b][1] * old[b][0]:
                    return None
            base = old[gi[-1]][1]
            acc = base
            for d in reversed(gj):
                new_st[d] = acc
                acc *= shape[d]
        return View(shape, new_st, self.offset, None)

    def max_offset(self):
        """Largest element offset an unmasked read can reach (for extents)."""
        if any(s == 0 for s in self.shape):
            return -1
        lo_hi = self._mask()
        off = self.offset
        for (lo, hi), s, t in zip(lo_hi, self.shape, self.strides):
            hi = min(hi, s)
            if hi <= max(lo, 0):
                return -1
            off += (hi - 1) * t
        return off
