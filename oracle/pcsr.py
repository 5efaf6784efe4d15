"""Padded-CSR reference state machine (TEST INFRASTRUCTURE ONLY).

Only the tests use this module; the CUDA library never does, and the two
share no code.  Plain Python lists, one operation at a time, in the order the
page describes them:

  "Padded-CSR: A sparse storage format for dynamic sparse training on CPU"
    sec. 5.1  the six arrays: slot values and column indices (-1 marks a
              padding slot), row_start, row_nnz (live slots come first in a
              row's region), row_capacity, topology_version;
    sec. 5.2  row_capacity = max(1, ceil(row_nnz * (1 + padding_ratio)));
    sec. 5.3  encoding of a matrix, and an insertion that writes the slot
              row_start + row_nnz and bumps the counter (O(1));
    sec. 4.3  a full row is resized: more slots are allocated, the row is
              copied and its pointers updated;
    sec. 8.3  compact_all: for adaptive-density DST (per-row nnz changes).

Readings where the page is silent (the library takes the same ones):
  * padding is a whole percentage p, and ceil(n * (100 + p) / 100) is taken
    in integers (the page's 0.2 is p = 20; every printed example agrees);
  * inserts come as a batch: a row whose live count plus its inserts exceeds
    its capacity is moved, before any insert is written, to fresh slots at the
    end of the used slot area with capacity max(1, ceil((live + inserted) *
    (100 + p) / 100)); rows move in ascending row order, their old slots become
    padding; then each insert takes the next free slot of its row, in batch
    order;
  * a delete clears the slot of (row, col) and the row's remaining live
    entries close up in their order, so live slots stay first; deleting a
    position that is not live is an error and changes nothing;
  * compact_all lays the rows out again from slot 0, in row order, with the
    capacity rule applied to the current counts and each row's entries sorted
    by column (the canonical order of sec. 4.1);
  * topology_version goes up by one for every insert batch, delete batch and
    compact_all that is applied.
"""
from __future__ import annotations


def capacity(n_live: int, pct: int) -> int:
    """sec. 5.2, in integers: max(1, ceil(n * (100 + pct) / 100))."""
    return max(1, (n_live * (100 + pct) + 99) // 100)


class PaddedCSR:
    def __init__(self, out_f: int, in_f: int, rows, cols, values, pct: int = 20):
        """Encode a COO triple (any order, no duplicates): sec. 5.1 steps 1-5."""
        self.out_f, self.in_f, self.pct = out_f, in_f, pct
        entries = sorted(zip((int(r) for r in rows), (int(c) for c in cols),
                             (float(v) for v in values)))
        per_row = [[] for _ in range(out_f)]
        for r, c, v in entries:
            per_row[r].append((c, v))
        self.row_nnz = [len(e) for e in per_row]
        self.row_capacity = [capacity(n, pct) for n in self.row_nnz]
        self.row_start, pos = [], 0
        for cap in self.row_capacity:
            self.row_start.append(pos)
            pos += cap
        self.slot_values = [0.0] * pos
        self.slot_cols = [-1] * pos
        for r, e in enumerate(per_row):
            for j, (c, v) in enumerate(e):
                self.slot_values[self.row_start[r] + j] = v
                self.slot_cols[self.row_start[r] + j] = c
        self.version = 1

    @property
    def used(self) -> int:
        return len(self.slot_cols)

    def insert(self, rows, cols, values):
        """One batch of inserts (see the module docstring for the order)."""
        rows = [int(r) for r in rows]
        demand = [0] * self.out_f
        for r in rows:
            demand[r] += 1
        for r in range(self.out_f):
            if self.row_nnz[r] + demand[r] > self.row_capacity[r]:
                new_cap = capacity(self.row_nnz[r] + demand[r], self.pct)
                start, n = self.row_start[r], self.row_nnz[r]
                live_v = self.slot_values[start:start + n]
                live_c = self.slot_cols[start:start + n]
                for s in range(start, start + self.row_capacity[r]):
                    self.slot_values[s], self.slot_cols[s] = 0.0, -1
                new_start = self.used
                self.slot_values += live_v + [0.0] * (new_cap - n)
                self.slot_cols += live_c + [-1] * (new_cap - n)
                self.row_start[r], self.row_capacity[r] = new_start, new_cap
        for r, c, v in zip(rows, cols, values):
            s = self.row_start[r] + self.row_nnz[r]
            self.slot_values[s], self.slot_cols[s] = float(v), int(c)
            self.row_nnz[r] += 1
        if rows:
            self.version += 1

    def delete(self, rows, cols):
        """One batch of deletes; raises KeyError (nothing changed) if a
        position is not live."""
        targets = []
        for r, c in zip(rows, cols):
            r, c = int(r), int(c)
            start = self.row_start[r]
            live = self.slot_cols[start:start + self.row_nnz[r]]
            if c not in live:
                raise KeyError((r, c))
            targets.append((r, start + live.index(c)))
        if not targets:
            return
        for r, s in targets:
            self.slot_cols[s] = -1
        for r in sorted({r for r, _ in targets}):
            start, n = self.row_start[r], self.row_nnz[r]
            kept = [(self.slot_cols[s], self.slot_values[s]) for s in range(start, start + n)
                    if self.slot_cols[s] != -1]
            for j in range(self.row_capacity[r]):
                c, v = kept[j] if j < len(kept) else (-1, 0.0)
                self.slot_cols[start + j], self.slot_values[start + j] = c, v
            self.row_nnz[r] = len(kept)
        self.version += 1

    def live_triple(self):
        """The live entries in canonical order (row, then column)."""
        out = []
        for r in range(self.out_f):
            s = self.row_start[r]
            for j in range(self.row_nnz[r]):
                out.append((r, self.slot_cols[s + j], self.slot_values[s + j]))
        out.sort()
        return ([e[0] for e in out], [e[1] for e in out], [e[2] for e in out])

    def compact_all(self):
        rows, cols, vals = self.live_triple()
        version = self.version
        self.__init__(self.out_f, self.in_f, rows, cols, vals, self.pct)
        self.version = version + 1
