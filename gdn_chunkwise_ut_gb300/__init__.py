"""kkt_solve for GB300: the chunk-local UT transform of Gated DeltaNet prefill."""
