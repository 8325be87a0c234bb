"""Plain, slow, obviously-correct CPU oracle for log-linear attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or call
anything in this package.  The product path (the C-ABI library and its Python
binding) never imports it, and this package imports nothing from the product.

Everything here is NumPy in float64.  Inputs arrive as arrays (callers pass the
bf16-rounded values upcast to float64 when the GPU path runs in bf16), so the
error measured against the GPU is compute error, not input quantisation.

Sources (page title, section):
  * "Log-Linear Attention" study note (dimensionstp.github.io):
      §1-2 (linear-attention recurrence), §2-2 (Fenwick partition, level
      states, output as a lambda-weighted sum over levels), §3-3 (recurrent
      form), §3-4 (parallel form O = (QK^T . M^H) V), §3-5 (mask composition
      M = M^S . M^H; Log-Linear Mamba-2 and Gated DeltaNet), §3-6 (decoding
      with O(log T) states tied to the bits of t).
  * gist.science "Log-Linear Attention" (zh), §2.2 and the drawer analogy
      (new token enters drawer 0; a full drawer merges into the next one).
  * gist.science "Log-Linear Attention" (de), Technische Zusammenfassung §2
      (output formula; Gated DeltaNet = delta rule combined with the
      hierarchical structure).

Readings taken where the pages are silent (each is stated where it is used):
  R1 level function l(t,s) = 0 if s == t else floor(log2(t xor s)) + 1;
  R3 the state at t includes token t (level 0);
  R4 M^S(t,s) = prod of alpha over (s, t], M^S(t,t) = 1;
  R7 Gated DeltaNet: the standard gated delta rule, with M^H applied to the
     full delta-rule coefficient matrix ("reading A"); "reading B" is also
     provided.  The pages do not fix which one the authors use: parity of A
     versus B is unpinned by the pages.
"""

from . import partition, mamba2, gdn, decode, backward, level_decay  # noqa: F401
