"""CPU oracle for the fusion-group hot path -- TEST INFRASTRUCTURE ONLY.

This package is the plain, slow, obviously correct statement of what the hot
path computes.  Only the test suite, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import it; the product path (the C-ABI library
and its Python binding) never does, and shares no code with it.

What it computes, and where the pages define it:

* a fusion group is evaluated node by node, one full intermediate array per
  node, every node in f32 and only the root rounded to its storage type
  (PSK-Realize, "What a group is"; "What it buys": fusion reassociates
  nothing) -- ``oracle.group``;
* the reduction-rooted softmax region Reduce(Max) -> Sub -> Exp ->
  Reduce(Sum) -> Div over the last axis, with the sum's bracketing tree fixed
  by the declared order (poot "Fusion and Planning", Reduction-rooted regions;
  presk "Native execution", The realization: ``order``) -- ``oracle.softmax``;
* the reduction-rooted normalization regions RMSNorm (sum of squares -> mean
  -> +eps -> sqrt -> divide) and LayerNorm (mean -> x - mu -> sum of squares
  -> mean -> +eps -> sqrt -> divide), with an optional scale and bias (poot
  "Fusion and Planning", Reduction-rooted regions; PSK-Realize, "What it
  removes") -- ``oracle.norm``;
* the AdamW step as PyTorch defines it, one f32 chain per parameter over every
  leaf of the tree (presk "The language", The optimizer) -- ``oracle.adamw``;
* exp and erf nodes return the correctly rounded f32 value of the function
  (``oracle.crmath``), and bf16 storage is a shift in and one round to
  nearest even out (presk "Native execution", bf16 is storage only) --
  ``oracle.f32``.

Every function is pinned by ``-m "not gpu"`` tests against values fixed by the
mathematics (exact rational arithmetic, an independent multiprecision library,
closed forms and invariants).
"""
