"""fp64 CPU oracle for the DeepSeek-V4-style compressed sparse attention layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library (no kernels, headers, tables or helpers) and it
imports nothing from ``compressed_sparse_long_c4a_gb300``.

Every function is a plain, slow, obviously-correct restatement of the method
described on the page "DeepSeek V4 in vLLM: Efficient Long-context Attention"
(vLLM blog, April 2026), computed in float64 with numpy.  Each module header
says which passage it follows and which readings it takes where the page is
silent.

Pinning status (what each part is checked against, in ``tests/``):
  formats     - exhaustive codec checks against torch.float8_e4m3fn and the
                OCP e2m1 value table; bf16 against torch.bfloat16; the MX
                power-of-two block scale by hand-worked blocks and its
                error bound; the DeepSeek-V4 584-byte row by the article's
                byte list and page formula, hand-worked scale bytes, a
                brute-force search for the scale rule, and its bytes
                against torch's e4m3 / bf16 casts.
  geometry    - closed forms for counts/windows/causality, brute-force
                enumeration of slot mapping.
  compressor  - closed forms (equal logits -> mean, dominant logit -> copy,
                RMS = 1), RoPE group identities, chunk == step.
  indexer     - brute-force sort on tiny inputs, all-tie rule, a hand-worked
                two-head score (ReLU, head weights).
  attention   - hand-worked two- and three-key examples (weights, values =
                keys, log-sum-exp), dense special case against torch fp64
                softmax + matmul, SWA coverage, translation invariance after
                inverse RoPE, a hand-worked inverse rotation.
  layer       - window keys rotated at their own positions (hand cos/sin
                values) and translation invariance of the whole chain
                (compress, window keys, attention, inverse RoPE) under a
                shift of every position by a multiple of 256.
  kvbytes     - the page's 9.62 GiB / 83.9 GiB / 8.7x figures.
  The page prints no worked numerical example; the hand examples above are
  computed from the definitions, not by this package.
"""
