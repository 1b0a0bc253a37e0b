"""CPU oracle for the speculative-decoding verify step (test infrastructure).

This package is test infrastructure only. It is a plain, slow, obviously
correct float64 restatement of what the verify step computes, written from
the pages on speculative decoding, and it shares no code with the CUDA path.
Only the test suite, the entry module's smoke check and the benchmark's CPU
baseline leg may import it; the product library never does.

Modules:
  philox   Philox4x32-10 counter RNG (Salmon, Moraes, Dror, Shaw, SC'11).
  w12      lossless 12-bit weight codec (SpecPilot digest, "Reasons").
  decoder  Llama-style decoder forward over a verify block (DSpark summary,
           "Architecture": the anchor + draft block verified in one pass).
  accept   greedy and rejection-sampling acceptance (LFM2.5-DSpark post,
           "Quality parity"; DSpark summary, "Problem").
  spec     autoregressive greedy decoding and the speculative loop used for
           token forcing (SpecPilot digest, intro).

Parity status: the decoder's logits are pinned only by special cases and
invariants (single-key attention, RoPE identity at position 0, uniform
attention through zero query/key weights, spec-greedy equal to AR-greedy);
no page prints a worked example of a forward pass. W12, Philox and both
acceptance rules are pinned by exhaustive, published or statistical checks.
"""
