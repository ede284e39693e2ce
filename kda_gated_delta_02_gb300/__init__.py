"""KDA (gated delta rule) hot path for GB300 -- Python binding placeholder."""
