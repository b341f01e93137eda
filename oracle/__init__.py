"""Plain CPU oracle for the three sequence-head relayouts.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package may import this
package; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use it.  It shares no code with the CUDA library.

Two independent oracles live here:

* ``oracle.loops`` -- scalar C loops (``vf_oracle.c``) whose loop nest is the
  destination layout, driven through ctypes;
* ``oracle.chain`` -- the pages' own reference mechanism, a PyTorch-CPU
  stack/split/permute/contiguous/cat materialisation ("Sol-Engine alignment on
  SM86 and SM89", section "What is enabled").

Parity status: pinned.  The tests pin both oracles to hand-derived worked
examples (``tests/golden/``), to the byte counts printed in the allocation
screen of the same section, to library routines in the P=1/C=1 special cases,
to a brute-force bijection on iota payloads, to the permutation invariant and
to round-trip identities; and the two oracles must agree bit for bit.

The opt-in lossy transport ("Sol-Engine alignment on SM86 and SM89", table
"Upstream gap and disposition", row "INT8 QKV and FP8 output transport") has
its oracle in the same C file (``oracle.loops.*_q``): the exact ops' loop
nests, quantising or dequantising one head row at a time.  Pinned: its scalar
conversions against PyTorch's float8_e4m3fn and bfloat16 conversions over
every code and tie, a row worked by hand, exact-grid rows whose codes must be
the exact layout and whose round trip must be bit-exact, and closed-form error
bounds.
"""
