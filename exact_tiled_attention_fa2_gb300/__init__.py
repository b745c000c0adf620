"""GB300-native exact tiled attention (FlashAttention-2 forward) for sm_103a."""
